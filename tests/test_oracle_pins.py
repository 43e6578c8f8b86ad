"""Pins for the fp64 oracle: each check is tied to something other than the
oracle itself -- a hand-worked example from the routing rules (golden/), a
closed form, brute force on tiny inputs, or a textbook reduction -- so that a
dropped term, a wrong sign or index, or a transposed operand fails one of them."""
import itertools
import json
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as W


def _golden(golden_dir, name):
    return json.loads((golden_dir / name).read_text())


# ---------------------------------------------------------------- router GEMM

def test_router_logits_exact_rational():
    """logits = x . Wr^T checked against an exact rational dot product."""
    rng = np.random.default_rng(7)
    T, E, H = 3, 5, 37
    x_bits = W.normal_bf16(11, 1, (T, H), 1.0)
    wr = rng.standard_normal((E, H)).astype(np.float32)
    got = oracle.router_logits(x_bits, wr)
    xf = W.bf16_to_f64(x_bits)
    for t in range(T):
        for e in range(E):
            exact = sum(Fraction(float(xf[t, h])) * Fraction(float(wr[e, h])) for h in range(H))
            assert abs(got[t, e] - float(exact)) <= 1e-13 * max(1.0, abs(float(exact)))
    # a transposed operand cannot silently pass: shapes are [T,E]
    assert got.shape == (T, E)


def _split_bound_ok(w32):
    hi, lo = oracle.split_router_weight(w32)
    w = w32.astype(np.float64)
    err = np.abs(w - (hi + lo / 256.0))
    # |W - W_high| <= half a bf16 ulp of W, and |256 r - W_low| <= half a bf16 ulp of 256 r
    # give |W - (W_high + W_low/256)| <= 2^-16 |W| (normal range).
    return err <= np.ldexp(np.abs(w), -16), hi, lo


def test_router_split_closed_form_bound_sweep():
    """Closed-form error bound of the two-BF16 split over a sweep of fp32 bit patterns
    covering every exponent of the normal range and 2^16 mantissas per exponent."""
    mant = np.arange(0, 1 << 23, 1 << 7, dtype=np.uint32)
    for exp in range(1, 200, 3):  # keep 256 * r inside the normal range
        bits = (np.uint32(exp) << np.uint32(23)) | mant
        for sign in (0, 1):
            w32 = (bits | np.uint32(sign << 31)).view(np.float32)
            ok, hi, lo = _split_bound_ok(w32)
            assert ok.all(), (exp, sign)


def test_router_split_is_round_to_nearest_even():
    """bf16 RNE on hand-picked patterns: ties go to the even mantissa."""
    def f(bits):
        return np.array([bits], dtype=np.uint32).view(np.float32)
    # 1 + 2^-8 is exactly half-way between bf16 1.0 and 1 + 2^-7: rounds to 1.0 (even)
    assert oracle.bf16_round(f(0x3F808000))[0] == 1.0
    # 1 + 3*2^-8 is half-way between 1 + 2^-7 (odd) and 1 + 2^-6: rounds up to 1 + 2^-6
    assert oracle.bf16_round(f(0x3F818000))[0] == 1.0 + 2.0 ** -6
    # just above the half-way point rounds up
    assert oracle.bf16_round(f(0x3F808001))[0] == 1.0 + 2.0 ** -7
    hi, lo = oracle.split_router_weight(f(0x3F808001))
    assert hi[0] == 1.0 + 2.0 ** -7
    # residual = (1 + 2^-8 + 2^-23) - (1 + 2^-7) = -2^-8 + 2^-23 ; x256 = -1 + 2^-15 -> bf16 -1
    assert lo[0] == -1.0


def test_router_split_logits_within_bound_of_exact():
    rng = np.random.default_rng(3)
    x = W.normal_bf16(5, 1, (8, 512), 1.0)
    wr = (rng.standard_normal((24, 512)) * 0.02).astype(np.float32)
    exact = oracle.router_logits(x, wr)
    hi, lo = oracle.split_router_weight(wr)
    approx = oracle.router_logits_split(x, hi, lo)
    bound = (np.abs(W.bf16_to_f64(x)) @ np.ldexp(np.abs(wr.astype(np.float64)), -16).T)
    assert (np.abs(approx - exact) <= bound + 1e-15).all()
    rel = np.linalg.norm(approx - exact) / np.linalg.norm(exact)
    assert rel < 1e-5


# ------------------------------------------------------- scoring / top-k / renorm

def test_silu_closed_form(golden_dir):
    g = _golden(golden_dir, "routing_worked_example.json")["silu"]
    np.testing.assert_allclose(oracle.silu(np.array(g["g"])), g["silu"], rtol=1e-15, atol=1e-16)
    # tails: SiLU(g) -> g for large g, -> 0 for very negative g
    assert oracle.silu(np.array([60.0]))[0] == pytest.approx(60.0, rel=1e-15)
    assert abs(oracle.silu(np.array([-800.0]))[0]) == 0.0


def test_sigmoid_routing_worked_examples(golden_dir):
    for case in _golden(golden_dir, "routing_worked_example.json")["sigmoid_cases"]:
        logits = np.array([case["logits"]])
        r = oracle.route_sigmoid(logits, np.array(case["bias"], dtype=np.float64), case["k"], case["route_scale"])
        assert r["idx"][0].tolist() == case["idx"], case["note"]
        np.testing.assert_allclose(r["w"][0], case["w"], rtol=1e-12)
        assert r["w"][0].sum() / case["route_scale"] == pytest.approx(case["w_unscaled_sum"], abs=1e-12)


def test_softmax_routing_worked_example(golden_dir):
    for case in _golden(golden_dir, "routing_worked_example.json")["softmax_cases"]:
        r = oracle.route_softmax(np.array([case["logits"]]), case["k"], case["eps"])
        assert r["idx"][0].tolist() == case["idx"]
        np.testing.assert_allclose(r["w"][0], case["w"], rtol=1e-12)


def _brute_topk(keys, k):
    """All k-subsets; the top-k set is the one whose every member beats every
    non-member, where 'beats' is (larger key) or (equal key and lower index)."""
    E = len(keys)

    def beats(a, b):
        return keys[a] > keys[b] or (keys[a] == keys[b] and a < b)

    winners = [s for s in itertools.combinations(range(E), k)
               if all(beats(a, b) for a in s for b in range(E) if b not in s)]
    assert len(winners) == 1
    return sorted(winners[0], key=lambda e: (-keys[e], e))


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(0)
    for trial in range(300):
        E = int(rng.integers(2, 8))
        k = int(rng.integers(1, E + 1))
        keys = rng.integers(0, 4, size=E).astype(np.float64) / 4.0  # many exact ties
        idx, margin = oracle.topk_desc(keys[None, :], k)
        assert idx[0].tolist() == _brute_topk(keys.tolist(), k)
        srt = sorted(keys, reverse=True)
        exp_margin = srt[k - 1] - srt[k] if k < E else math.inf
        assert margin[0] == exp_margin


def test_renormalised_weights_sum():
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((64, 192)) * 1.3
    bias = rng.standard_normal(192) * 0.1
    r1 = oracle.route_sigmoid(logits, bias, 8, 1.0)
    np.testing.assert_allclose(r1["w"].sum(1), 1.0, atol=1e-12)
    r2 = oracle.route_sigmoid(logits, bias, 8, 2.826)
    np.testing.assert_allclose(r2["w"].sum(1), 2.826, atol=1e-12)
    # the weights are the unbiased sigmoids, not the biased keys
    s = 1.0 / (1.0 + np.exp(-logits))
    sel = np.take_along_axis(s, r2["idx"].astype(np.int64), 1)
    np.testing.assert_allclose(r2["w"], sel / sel.sum(1, keepdims=True) * 2.826, rtol=1e-14)


def test_bias_changes_selection_never_weights():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((32, 16))
    bias = rng.standard_normal(16) * 0.1
    r = oracle.route_sigmoid(logits, bias, 4, 2.826)
    # a bias shift that keeps every row's key order keeps the selection; weights identical
    r_shift = oracle.route_sigmoid(logits, bias + 5.0, 4, 2.826)
    assert np.array_equal(r["idx"], r_shift["idx"])
    assert np.array_equal(r["w"], r_shift["w"])
    # a bias that reorders changes the selection, and the weights are the unbiased
    # sigmoids of the new selection
    big = np.zeros(16)
    big[[3, 5, 7, 9]] = 10.0
    r_big = oracle.route_sigmoid(logits, big, 4, 2.826)
    assert (np.sort(r_big["idx"], 1) == np.array([3, 5, 7, 9])).all()
    s = 1.0 / (1.0 + np.exp(-logits[:, [3, 5, 7, 9]]))
    np.testing.assert_allclose(np.sort(r_big["w"], 1), np.sort(s / s.sum(1, keepdims=True) * 2.826, 1), rtol=1e-14)


def test_softmax_topk_equals_softmax_over_selected():
    """Closed form: top-k of a softmax renormalised = softmax over the k selected logits."""
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((50, 64)) * 2.0
    r = oracle.route_softmax(logits, 8, 1e-8)
    sel = np.take_along_axis(logits, r["idx"].astype(np.int64), 1)
    closed = np.exp(sel - sel.max(1, keepdims=True))
    closed /= closed.sum(1, keepdims=True)
    np.testing.assert_allclose(r["w"], closed, rtol=1e-12)
    np.testing.assert_allclose(r["w"].sum(1), 1.0, atol=1e-13)
    # selection on the softmax equals selection on the logits (monotone)
    idx2, _ = oracle.topk_desc(logits, 8)
    assert np.array_equal(r["idx"], idx2)


def test_clamp_degenerate_case():
    """The clamp only acts when the selected mass is below eps."""
    sel = np.array([[2e-9, 3e-9], [0.2, 0.3]])
    w = oracle.renormalize(sel, 1e-8)
    np.testing.assert_allclose(w[0], [0.2, 0.3], rtol=1e-15)
    np.testing.assert_allclose(w[1], [0.4, 0.6], rtol=1e-15)


def test_near_tie_alternatives():
    keys = np.array([[0.9, 0.5, 0.5 + 4e-6, 0.1, 0.5 - 3e-6]])
    mand, cand = oracle.near_tie_alternatives(keys, 2, 1e-5)
    assert mand[0].tolist() == [True, False, False, False, False]
    assert cand[0].tolist() == [False, True, True, False, True]


# ------------------------------------------- a given selection (near-tie rows)
# The GPU parity tests grade a near-tie row against the oracle re-evaluated with
# the GPU's selection (layer_forward(topk_idx=...)); these pins tie that path to
# hand-worked weights, so a wrong weight rule for a given selection fails here.

def _override_cases(golden_dir):
    return _golden(golden_dir, "routing_worked_example.json")["override_cases"]


def _one_token_layer(case, seed=31, I=3, Is=2):
    """One token whose router logits are the case's logits: H = 1, hidden [[1.0]]
    (bf16 0x3F80) and a one-column fp32 router weight holding the logits."""
    E = len(case["logits"])
    x = np.array([[0x3F80]], dtype=np.uint16)
    wr = np.array(case["logits"], dtype=np.float32)[:, None]
    bias = np.array(case["bias"], dtype=np.float32) if case["mode"] == "sigmoid" else None
    wg = W.normal_bf16(seed, 4, (E, I, 1), 0.7)
    wu = W.normal_bf16(seed, 5, (E, I, 1), 0.7)
    wd = W.normal_bf16(seed, 6, (E, 1, I), 0.7)
    sg = W.normal_bf16(seed, 7, (Is, 1), 0.7)
    su = W.normal_bf16(seed, 8, (Is, 1), 0.7)
    sd = W.normal_bf16(seed, 9, (1, Is), 0.7)
    return x, wr, bias, wg, wu, wd, sg, su, sd


def _run_case(case, inputs, topk_idx=None):
    return oracle.layer_forward(*inputs, top_k=case["k"], score_mode=case["mode"], route_scale=case["route_scale"],
                                renorm_eps=case["eps"], topk_idx=topk_idx)


def test_given_selection_weights_hand_worked(golden_dir):
    """A valid alternative selection gets the weights the routing rule gives that
    set: the unbiased sigmoids renormalised and scaled (sigmoid rule), or the
    softmax mass over clamp(sum, eps) (softmax rule) -- not the biased keys, not
    the unscaled sum, not the unclamped sum."""
    for case in _override_cases(golden_dir):
        inputs = _one_token_layer(case)
        own = _run_case(case, inputs)
        assert own["idx"][0].tolist() == case["own_idx"], case["note"]
        np.testing.assert_allclose(own["w"][0], case["own_w"], rtol=1e-6)
        # the alternative is a valid near-tie choice under the 1e-5 rule
        mand, cand = oracle.near_tie_alternatives(own["keys"], case["k"], 1e-5)
        alt = set(case["alt_idx"])
        assert set(np.nonzero(mand[0])[0]) <= alt <= set(np.nonzero(mand[0] | cand[0])[0])
        r = _run_case(case, inputs, topk_idx=np.array([case["alt_idx"]], dtype=np.int32))
        assert r["idx"][0].tolist() == case["alt_idx"]
        np.testing.assert_allclose(r["w"][0], case["alt_w"], rtol=1e-6)


def test_given_selection_layer_matches_per_token_brute_force(golden_dir):
    """The layer output for the alternative selection equals a direct per-token
    sum of the chosen experts' SwiGLU outputs with the hand-worked weights, plus
    the shared expert."""
    f = W.bf16_to_f64
    for case in _override_cases(golden_dir):
        inputs = _one_token_layer(case)
        x, _, _, wg, wu, wd, sg, su, sd = inputs
        r = _run_case(case, inputs, topk_idx=np.array([case["alt_idx"]], dtype=np.int32))
        out = _dense_swiglu_loops(f(x), f(sg), f(su), f(sd))[0]
        for e, w in zip(case["alt_idx"], case["alt_w"]):
            out = out + w * _dense_swiglu_loops(f(x), f(wg[e]), f(wu[e]), f(wd[e]))[0]
        np.testing.assert_allclose(r["out"][0], out, rtol=1e-6, atol=1e-12)


@pytest.mark.parametrize("mode", ["sigmoid", "softmax"])
def test_given_own_selection_is_the_default_call(mode):
    """Passing the oracle's own selection back in changes nothing, bit for bit."""
    T, H, E, k, I, Is = 9, 8, 6, 3, 4, 5
    x, wr, b, wg, wu, wd, sg, su, sd = _tiny_layer_inputs(24, T, H, E, I, Is)
    kw = dict(top_k=k, score_mode=mode, route_scale=2.826 if mode == "sigmoid" else 1.0,
              renorm_eps=0.0 if mode == "sigmoid" else 1e-8)
    r = oracle.layer_forward(x, wr, b, wg, wu, wd, sg, su, sd, **kw)
    r2 = oracle.layer_forward(x, wr, b, wg, wu, wd, sg, su, sd, topk_idx=r["idx"], **kw)
    for key in ("idx", "w", "perm", "inv", "out"):
        assert np.array_equal(r[key], r2[key]), key


# --------------------------------------------------------- histogram / permutation

def test_permutation_brute_force_and_invariants():
    rng = np.random.default_rng(5)
    for trial in range(50):
        T, E = int(rng.integers(1, 20)), int(rng.integers(1, 9))
        k = int(rng.integers(1, E + 1))
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        counts, offsets = oracle.histogram_offsets(idx, E)
        perm, inv = oracle.permutation(idx, E)
        S = T * k
        assert counts.sum() == S and offsets[-1] == S and offsets[0] == 0
        assert sorted(perm.tolist()) == list(range(S))          # bijection
        assert (inv[perm] == np.arange(S)).all() and (perm[inv] == np.arange(S)).all()
        # brute force: stable sort of slots by (expert, slot)
        flat = idx.reshape(-1).tolist()
        expected = sorted(range(S), key=lambda s: (flat[s], s))
        assert perm.tolist() == expected
        for e in range(E):
            seg = perm[offsets[e]:offsets[e + 1]]
            assert all(flat[s] == e for s in seg) and list(seg) == sorted(seg)
            assert counts[e] == flat.count(e)


# ------------------------------------------------------------- expert FFN / layer

def _dense_swiglu_loops(x, wg, wu, wd):
    """Independently written dense SwiGLU with explicit index loops:
    g_i = sum_h Wg[i,h] x_h ; u_i = sum_h Wu[i,h] x_h ; a_i = g_i/(1+e^-g_i) u_i ;
    y_o = sum_i Wd[o,i] a_i."""
    T, H = x.shape
    I = wg.shape[0]
    y = np.zeros((T, wd.shape[0]))
    for t in range(T):
        a = []
        for i in range(I):
            g = sum(float(wg[i, h]) * float(x[t, h]) for h in range(H))
            u = sum(float(wu[i, h]) * float(x[t, h]) for h in range(H))
            a.append(g / (1.0 + math.exp(-g)) * u)
        for o in range(wd.shape[0]):
            y[t, o] = sum(float(wd[o, i]) * a[i] for i in range(I))
    return y


def _tiny_layer_inputs(seed, T, H, E, I, Is):
    x = W.normal_bf16(seed, 1, (T, H), 1.0)
    wr = W.normal_f32(seed, 2, (E, H), 0.3)
    b = W.normal_f32(seed, 3, (E,), 0.1)
    wg = W.normal_bf16(seed, 4, (E, I, H), 0.3)
    wu = W.normal_bf16(seed, 5, (E, I, H), 0.3)
    wd = W.normal_bf16(seed, 6, (E, H, I), 0.3)
    sg = W.normal_bf16(seed, 7, (Is, H), 0.3)
    su = W.normal_bf16(seed, 8, (Is, H), 0.3)
    sd = W.normal_bf16(seed, 9, (H, Is), 0.3)
    return x, wr, b, wg, wu, wd, sg, su, sd


def test_dense_reduction_E1_k1():
    """E = 1, k = 1: the layer is route_scale x one dense SwiGLU (+ the shared MLP)."""
    T, H, I, Is = 3, 6, 5, 4
    x, wr, b, wg, wu, wd, sg, su, sd = _tiny_layer_inputs(21, T, H, 1, I, Is)
    f = W.bf16_to_f64
    dense = _dense_swiglu_loops(f(x), f(wg[0]), f(wu[0]), f(wd[0]))
    shared = _dense_swiglu_loops(f(x), f(sg), f(su), f(sd))
    r = oracle.layer_forward(x, wr, b, wg, wu, wd, None, None, None, top_k=1, route_scale=2.826)
    np.testing.assert_allclose(r["out"], 2.826 * dense, rtol=1e-12, atol=1e-12)
    r = oracle.layer_forward(x, wr, b, wg, wu, wd, sg, su, sd, top_k=1, route_scale=2.826)
    np.testing.assert_allclose(r["out"], 2.826 * dense + shared, rtol=1e-12, atol=1e-12)
    r = oracle.layer_forward(x, wr, None, wg, wu, wd, sg, su, sd, top_k=1, score_mode="softmax",
                             route_scale=1.0, renorm_eps=1e-8)
    np.testing.assert_allclose(r["out"], dense + shared, rtol=1e-12, atol=1e-12)


def test_layer_matches_per_token_brute_force():
    """Whole layer on a tiny case against per-token loops over the selected experts."""
    T, H, E, k, I, Is = 5, 6, 4, 2, 3, 5
    x, wr, b, wg, wu, wd, sg, su, sd = _tiny_layer_inputs(22, T, H, E, I, Is)
    f = W.bf16_to_f64
    r = oracle.layer_forward(x, wr, b, wg, wu, wd, sg, su, sd, top_k=k, route_scale=2.826)
    for t in range(T):
        logits = [sum(float(f(x)[t, h]) * float(wr[e, h]) for h in range(H)) for e in range(E)]
        s = [1.0 / (1.0 + math.exp(-v)) for v in logits]
        keys = [s[e] + float(b[e]) for e in range(E)]
        chosen = _brute_topk(keys, k)
        tot = sum(s[e] for e in chosen)
        out = _dense_swiglu_loops(f(x)[t:t + 1], f(sg), f(su), f(sd))[0]
        for e in chosen:
            out = out + (s[e] / tot * 2.826) * _dense_swiglu_loops(f(x)[t:t + 1], f(wg[e]), f(wu[e]), f(wd[e]))[0]
        np.testing.assert_allclose(r["out"][t], out, rtol=1e-11, atol=1e-12)


def test_permutation_equivariance():
    T, H, E, k, I, Is = 12, 8, 6, 3, 4, 4
    x, wr, b, wg, wu, wd, sg, su, sd = _tiny_layer_inputs(23, T, H, E, I, Is)
    r = oracle.layer_forward(x, wr, b, wg, wu, wd, sg, su, sd, top_k=k)
    p = np.random.default_rng(9).permutation(T)
    rp = oracle.layer_forward(x[p], wr, b, wg, wu, wd, sg, su, sd, top_k=k)
    np.testing.assert_allclose(rp["out"], r["out"][p], rtol=1e-13, atol=1e-13)
    # and a sample of rows equals the same rows of the full batch
    rows = oracle.layer_rows(x[[2, 7]], wr, b, wg, wu, wd, sg, su, sd, top_k=k)
    np.testing.assert_allclose(rows["out"], r["out"][[2, 7]], rtol=1e-13, atol=1e-13)


def test_combine_brute_force():
    rng = np.random.default_rng(6)
    T, k, H = 4, 3, 5
    y = rng.standard_normal((T * k, H))
    z = rng.standard_normal((T, H))
    w = rng.random((T, k))
    inv = rng.permutation(T * k).astype(np.int32)
    out = oracle.combine(y, inv, w, z)
    for t in range(T):
        for h in range(H):
            ref = z[t, h] + sum(w[t, j] * y[inv[t * k + j], h] for j in range(k))
            assert out[t, h] == pytest.approx(ref, rel=1e-14, abs=1e-14)


def test_expert_outputs_sorted_rows():
    """y_sorted[p] is the FFN of expert e applied to token perm[p] // k."""
    T, H, E, k, I = 7, 6, 3, 2, 4
    x, wr, b, wg, wu, wd, _, _, _ = _tiny_layer_inputs(24, T, H, E, I, 2)
    idx = np.array([[0, 2], [1, 0], [2, 1], [0, 1], [2, 0], [1, 2], [0, 2]], dtype=np.int32)
    counts, offsets = oracle.histogram_offsets(idx, E)
    perm, inv = oracle.permutation(idx, E)
    y = oracle.expert_outputs_sorted(x, perm, offsets, k, wg, wu, wd)
    f = W.bf16_to_f64
    for p in range(T * k):
        t, j = divmod(int(perm[p]), k)
        e = int(idx[t, j])
        ref = _dense_swiglu_loops(f(x)[t:t + 1], f(wg[e]), f(wu[e]), f(wd[e]))[0]
        np.testing.assert_allclose(y[p], ref, rtol=1e-12, atol=1e-13)


def test_model_facts_match_workloads(golden_dir):
    facts = _golden(golden_dir, "model_facts.json")
    d = W.WORKLOADS["decode"]
    hy3 = facts["hy3"]
    assert (d.H, d.E, d.top_k, d.I, d.route_scale) == (
        hy3["hidden_size"], hy3["routed_experts"], hy3["top_k"], hy3["expert_intermediate"],
        hy3["router_scaling_factor"])
    img = W.WORKLOADS["image"]
    hi = facts["hunyuan_image"]
    assert (img.H, img.E, img.I, img.renorm_eps, img.score_mode) == (
        hi["hidden_size"], hi["routed_experts"], hi["expert_intermediate"], hi["clamp_min"], hi["score"])
    assert facts["router_split"]["scale"] == 1.0 / 256.0


# ---------------------------------------------------------------- FP8 (E4M3) expert weights
# The format is the OCP 8-bit floating point specification's E4M3: its table of
# special values gives the constants below (max normal S.1111.110 = 448, min
# normal S.0001.000 = 2^-6, max subnormal S.0000.111 = 0.875 * 2^-6, min
# subnormal S.0000.001 = 2^-9, S.1111.111 = NaN, no infinities).

def test_e4m3_special_values():
    v = oracle.e4m3_value(np.arange(256))
    exact = {0x00: Fraction(0), 0x01: Fraction(1, 2 ** 9), 0x07: Fraction(7, 8) / 2 ** 6, 0x08: Fraction(1, 2 ** 6),
             0x38: Fraction(1), 0x7E: Fraction(448), 0xB8: Fraction(-1), 0xFE: Fraction(-448)}
    for c, x in exact.items():
        assert Fraction(float(v[c])) == x, hex(c)
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF]) and np.isnan(v).sum() == 2
    assert v[0x80] == 0.0 and np.signbit(v[0x80])
    pos = v[:0x7F]
    assert (np.diff(pos) > 0).all()                      # codes 0x00..0x7E increase
    assert np.array_equal(v[0x80:0xFF], -pos)             # sign-magnitude
    # spacing: 2^-9 below 2^-5, then doubling at every binade (3 mantissa bits)
    gaps = np.diff(pos)                                   # gaps[c] = value(c + 1) - value(c)
    assert np.all(gaps[:8] == 2.0 ** -9)                 # subnormals and into the first binade
    for e in range(1, 16):                                # codes 8e .. 8e + 7 span binade e
        assert np.all(gaps[8 * e:8 * e + 8] == 2.0 ** (e - 10)), e


def _encode_brute(x):
    """Nearest of the 127 non-negative finite values by exhaustive search; a tie
    goes to the even code; past 448 the magnitude is clamped to 448."""
    pos = oracle.e4m3_value(np.arange(0x7F))
    if np.isnan(x):
        return 0x7F
    a = min(abs(x), 448.0)
    d = np.abs(pos - a)
    best = np.flatnonzero(d == d.min())
    c = int(best[0]) if len(best) == 1 else int(next(b for b in best if b % 2 == 0))
    return c | (0x80 if math.copysign(1.0, x) < 0 else 0)


def test_e4m3_encode_brute_force_ties_and_saturation():
    pos = oracle.e4m3_value(np.arange(0x7F))
    mids = (pos[:-1] + pos[1:]) / 2                        # exact ties between neighbours
    rng = np.random.default_rng(5)
    rand = np.concatenate([rng.standard_normal(2000) * s for s in (1e-3, 0.05, 1.0, 30.0, 300.0)])
    vals = np.concatenate([pos, -pos, mids, -mids, rand, [500.0, -1e9, 448.0 + 15.9, 0.0, -0.0, np.nan]])
    got = oracle.e4m3_encode(vals)
    want = np.array([_encode_brute(float(x)) for x in vals], dtype=np.uint8)
    assert np.array_equal(got, want)
    # every finite code survives decode -> encode
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_value(codes)), codes.astype(np.uint8))


def test_quantize_rows_bounds_and_zero_rows():
    rng = np.random.default_rng(9)
    w = W.normal_bf16(3, 7, (6, 256), 0.02)
    w[2] = 0                                             # an all-zero row: scale 1, codes 0
    q, s = oracle.quantize_rows_e4m3(w)
    wf = W.bf16_to_f64(w)
    assert s[2] == 1.0 and not q[2].any()
    for r in (0, 1, 3, 4, 5):
        assert s[r] == np.float32(np.float32(np.abs(wf[r]).max()) / np.float32(448.0))
        assert int((q[r] & 0x7F).max()) == 0x7E           # the row maximum lands on 448
    deq = oracle.dequantize_rows_e4m3(q, s)
    # E4M3 keeps 3 fraction bits: relative error <= 2^-4 on normals (plus the
    # fp32 division's half ulp), absolute <= 2^-10 * scale on subnormals
    err = np.abs(deq - wf)
    bound = np.maximum(np.abs(wf) * (2.0 ** -4 + 2.0 ** -20), s[:, None].astype(np.float64) * 2.0 ** -10 * 1.01)
    assert (err <= bound).all()


def test_fp8_weights_on_the_grid_reduce_to_the_bf16_layer():
    """Rows whose entries are E4M3 values times 2^-12 with the row maximum 448 *
    2^-12 quantise with scale 2^-12 and dequantise back exactly, so the layer on
    the dequantised weights is the bf16 layer bit for bit."""
    rng = np.random.default_rng(4)
    codes = rng.integers(0, 0x7F, size=(2, 16, 64)).astype(np.uint8)
    codes[..., 0] = 0x7E
    codes = codes | (rng.integers(0, 2, size=codes.shape).astype(np.uint8) << 7)
    w = oracle.e4m3_value(codes) * 2.0 ** -12
    q, s = oracle.quantize_rows_e4m3(w.astype(np.float32))
    assert np.all(s == np.float32(2.0 ** -12))
    assert np.array_equal(oracle.dequantize_rows_e4m3(q, s), w)


# ------------------------------------------------------------------- W8A8 (FP8 activations)

def _e4m3_decode(code):
    """E4M3 value from the bit fields of the OCP 8-bit format: sign, 4 exponent
    bits (bias 7, 0 = subnormal), 3 mantissa bits; S.1111.111 is NaN."""
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 15 and m == 7:
        return math.nan
    return sign * (m / 8.0 * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7))


_E4M3_TABLE = [(c, _e4m3_decode(c)) for c in range(256) if not math.isnan(_e4m3_decode(c))]


def _quantize_row_brute(row):
    """One row: scale = fp32(max|v|) / 448 in fp32 (1 for a zero row); each code the
    nearest E4M3 value to fp32(v) / scale (fp32 division), ties to the even code,
    by search over every code; magnitudes past 448 go to +-448."""
    r32 = np.asarray(row, dtype=np.float32)
    amax = np.float32(np.abs(r32).max())
    scale = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
    codes = []
    for v in (r32 / scale).astype(np.float32):
        v = float(v)
        best = min(_E4M3_TABLE, key=lambda cv: (abs(cv[1] - v), cv[0] & 1, cv[0]))
        codes.append(best[0])
    return codes, float(scale)


def _bf16_torch(x):
    import torch
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def _swiglu_w8a8_loops(x_row, g, u, d):
    """One token through one W8A8 SwiGLU expert with explicit index loops."""
    xq, xs = _quantize_row_brute(x_row)
    (gq, gs), (uq, us), (dq, ds) = g, u, d
    I, H = gq.shape
    a = []
    for i in range(I):
        gi = sum(_e4m3_decode(int(xq[h])) * _e4m3_decode(int(gq[i, h])) for h in range(H)) * xs * float(gs[i])
        ui = sum(_e4m3_decode(int(xq[h])) * _e4m3_decode(int(uq[i, h])) for h in range(H)) * xs * float(us[i])
        a.append(gi / (1.0 + math.exp(-gi)) * ui)
    a16 = _bf16_torch(np.array(a))
    aq, a_s = _quantize_row_brute(a16)
    out = []
    for o in range(dq.shape[0]):
        out.append(sum(_e4m3_decode(int(aq[i])) * _e4m3_decode(int(dq[o, i])) for i in range(I)) * a_s * float(ds[o]))
    return np.array(out)


def _w8a8_tiny(seed, T, H, E, I, Is):
    x, wr, b, wg, wu, wd, sg, su, sd = _tiny_layer_inputs(seed, T, H, E, I, Is)
    q = oracle.quantize_rows_e4m3
    experts = (q(wg), q(wu), q(wd))
    shared = (q(sg), q(su), q(sd))
    return x, wr, b, experts, shared, (wg, wu, wd, sg, su, sd)


def test_w8a8_swiglu_matches_index_loops():
    """One expert: quantised input row, gate/up from code products and both row
    scales, bf16 activation quantised per row, down projection -- against
    independently written loops."""
    x, _, _, experts, shared, _ = _w8a8_tiny(41, 4, 12, 2, 7, 5)
    xq, xs = oracle.quantize_rows_e4m3(x)
    (gq, gs), (uq, us), (dq, ds) = experts
    got = oracle.swiglu_w8a8(xq, xs, (gq[1], gs[1]), (uq[1], us[1]), (dq[1], ds[1]))
    f = W.bf16_to_f64
    for t in range(x.shape[0]):
        ref = _swiglu_w8a8_loops(f(x)[t], (gq[1], gs[1]), (uq[1], us[1]), (dq[1], ds[1]))
        np.testing.assert_allclose(got[t], ref, rtol=1e-12, atol=1e-14)


def test_w8a8_layer_matches_per_token_brute_force():
    T, H, E, k, I, Is = 5, 10, 4, 2, 6, 3
    x, wr, b, experts, shared, _ = _w8a8_tiny(42, T, H, E, I, Is)
    r = oracle.layer_forward_w8a8(x, wr, b, experts, shared, top_k=k, route_scale=2.826)
    ref_route = oracle.layer_forward(x, wr, b, *_tiny_layer_inputs(42, T, H, E, I, Is)[3:], top_k=k)
    assert np.array_equal(r["idx"], ref_route["idx"]) and np.array_equal(r["w"], ref_route["w"])
    f = W.bf16_to_f64
    (gq, gs), (uq, us), (dq, ds) = experts
    for t in range(T):
        out = _swiglu_w8a8_loops(f(x)[t], *shared)
        for j, e in enumerate(r["idx"][t]):
            out = out + r["w"][t, j] * _swiglu_w8a8_loops(f(x)[t], (gq[e], gs[e]), (uq[e], us[e]), (dq[e], ds[e]))
        np.testing.assert_allclose(r["out"][t], out, rtol=1e-11, atol=1e-13)


def test_w8a8_is_close_to_the_bf16_layer():
    """Quantisation noise only: E4M3 keeps 3 mantissa bits (relative spacing
    2^-3, rounding error <= 2^-4), so on Gaussian data the W8A8 layer stays
    within a few percent of the exact layer on the bf16 weights."""
    T, H, E, k, I, Is = 24, 64, 6, 2, 32, 32
    x, wr, b, experts, shared, raw = _w8a8_tiny(43, T, H, E, I, Is)
    r8 = oracle.layer_forward_w8a8(x, wr, b, experts, shared, top_k=k)
    r16 = oracle.layer_forward(x, wr, b, *raw, top_k=k)
    rel = np.linalg.norm(r8["out"] - r16["out"]) / np.linalg.norm(r16["out"])
    assert 1e-4 < rel < 0.08, rel
