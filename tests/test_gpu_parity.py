"""GPU parity: every stage of the CUDA path, called through the C ABI, against
the fp64 oracle on the same seeded inputs.

Small and medium shapes are compared element by element (several tiles and a
ragged tail); the full workload shapes are compared on sampled tokens (the
oracle computes them one by one) plus properties that hold at any size."""
import numpy as np
import pytest
import torch

import expert_ffn_layer_gb300 as moe
import oracle
import workloads as W
from moe_testlib import (LAYER_MAX_ABS, LAYER_REL_L2, NEAR_TIE, ROUTER_REL_L2, DeviceLayer, assert_layer_close,
                         bf16_dev, check_selection, dims_of, f32_dev, host_f64, i32_dev, oracle_layer, rel_l2,
                         valid_alternatives)

pytestmark = pytest.mark.gpu

# Medium shapes the oracle finishes in seconds: several router m-tiles with a
# ragged tail (T = 300), shared segment longer than one 256-token chunk, etc.
MID = W.Workload("mid", 300, 512, 8, 2, 256, 128, "sigmoid", 2.826, 0.0, True, "normal", 0.1, 5)
MID_SOFTMAX = W.Workload("mid_softmax", 300, 512, 16, 4, 256, 256, "softmax", 1.0, 1e-8, True, "none", 0.0, 6)
WIDE = W.Workload("wide", 64, 256, 256, 16, 64, 64, "sigmoid", 2.826, 0.0, True, "normal", 0.1, 7)
DENSE = W.Workload("dense", 37, 256, 1, 1, 128, 128, "sigmoid", 2.826, 0.0, True, "normal", 0.1, 8)
ODD_H = W.Workload("odd_h", 20, 192, 4, 2, 64, 64, "sigmoid", 2.826, 0.0, True, "normal", 0.1, 9)
NOSHARED = W.WORKLOADS["tiny"].with_(name="noshared", has_shared=False)
# 32 tokens at top-16 over 64 experts: 512 routed slots, the permutation's
# one-CTA form with every warp holding whole rounds of slots
SMALL32 = W.Workload("small32", 32, 512, 64, 16, 128, 128, "sigmoid", 2.826, 0.0, True, "normal", 0.1, 11)
SMALL = [W.WORKLOADS["tiny"], MID, MID_SOFTMAX, WIDE, DENSE, ODD_H, NOSHARED]
SMALL_IDS = [w.name for w in SMALL]


@pytest.fixture(scope="session", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


_cache = {}


def inputs_of(w):
    """Seeded inputs of a workload; the two most recent ones stay cached."""
    if w.name not in _cache:
        while len(_cache) >= 2:
            _cache.pop(next(iter(_cache)))
        _cache[w.name] = W.layer_inputs(w)
    return _cache[w.name]


def _ref_route(w, inp):
    logits = oracle.router_logits(inp["hidden"], inp["router_w"])
    if w.score_mode == "sigmoid":
        r = oracle.route_sigmoid(logits, inp["bias"], w.top_k, w.route_scale)
    else:
        r = oracle.route_softmax(logits, w.top_k, w.renorm_eps)
    r["logits"] = logits
    return r


def _check_route(w, inp, dl):
    idx, wts, logits = dl.route()
    torch.cuda.synchronize()
    ref = _ref_route(w, inp)
    lg = logits.cpu().numpy().astype(np.float64)
    assert rel_l2(lg, ref["logits"]) <= ROUTER_REL_L2, rel_l2(lg, ref["logits"])
    gi = idx.cpu().numpy()
    gw = wts.cpu().numpy().astype(np.float64)
    same, ties = check_selection(gi, ref, w.top_k)
    # keys are in descending order in the GPU output: weights of the same experts must match
    for t in same:
        o = dict(zip(ref["idx"][t].tolist(), ref["w"][t].tolist()))
        for j, e in enumerate(gi[t].tolist()):
            assert abs(gw[t, j] - o[e]) <= 2e-4 * max(1.0, w.route_scale), (t, e, gw[t, j], o[e])
    for t in ties:
        alt = oracle.routing_weights_for(ref["scores"][t:t + 1], np.sort(gi[t:t + 1], 1), w.score_mode,
                                         w.route_scale, w.renorm_eps)[0]
        np.testing.assert_allclose(np.sort(gw[t]), np.sort(alt), atol=2e-4 * max(1.0, w.route_scale))
    if getattr(dl, "ws", None) is not None:
        assert moe.moe_ws_read_error(dl.ws) == 0
    # descending key order inside a row (ties: lower expert first)
    k_of = ref["keys"]
    for t in same[:64]:
        ks = [k_of[t, e] for e in gi[t]]
        assert all(ks[j] >= ks[j + 1] - NEAR_TIE for j in range(len(ks) - 1))
    return gi, ref, ties


# ------------------------------------------------------------------ router

@pytest.mark.parametrize("w", SMALL + [W.WORKLOADS["decode"]], ids=SMALL_IDS + ["decode"])
def test_route_parity(w):
    inp = inputs_of(w) if w.name != "decode" else None
    if inp is None:  # the router needs no expert weights
        hidden, router_w, bias = W.router_inputs(w)
        inp = {"hidden": hidden, "router_w": router_w, "bias": bias}
        d = dims_of(w)
        dl = type("R", (), {})()
        dl.d = d
        dl.hidden, dl.router_w, dl.bias = bf16_dev(hidden), f32_dev(router_w), f32_dev(bias)
        dl.ws = moe.alloc_workspace(d)
        dl.route = lambda: DeviceLayer.route(dl)
    else:
        dl = DeviceLayer(w, inp)
    _check_route(w, inp, dl)


def _router_only(w):
    """Device inputs of the router alone (no expert weights)."""
    hidden, router_w, bias = W.router_inputs(w)
    inp = {"hidden": hidden, "router_w": router_w, "bias": bias}
    dl = type("R", (), {})()
    dl.d = dims_of(w)
    dl.hidden, dl.router_w, dl.bias = bf16_dev(hidden), f32_dev(router_w), f32_dev(bias)
    dl.ws = moe.alloc_workspace(dl.d)
    dl.route = lambda: DeviceLayer.route(dl)
    return inp, dl


@pytest.mark.parametrize("T,H,E,k,mode", [(128, 1024, 192, 8, "sigmoid"), (129, 1024, 192, 8, "sigmoid"),
                                          (100, 512, 256, 8, "softmax"), (1, 4096, 192, 8, "sigmoid"),
                                          (77, 640, 48, 6, "sigmoid"), (32, 4096, 192, 8, "sigmoid"),
                                          (32, 512, 256, 16, "softmax"), (33, 4096, 192, 8, "sigmoid"),
                                          (4100, 1024, 192, 8, "sigmoid"), (4100, 1024, 64, 8, "softmax")])
def test_route_one_tile_and_boundary(T, H, E, k, mode):
    """A full 128-token tile, one token more (a second tile of one row), a
    single token, E = 256 (one 256-column accumulator pair), and H = 640 (ten K
    slices: a split of two); 32 and 33 tokens at the Hy3 shape, and 32 tokens
    with E = 256 and top-16; 4100 tokens (the top-k kernel's eight-token CTAs,
    four K slices, a ragged last tile) in both scoring modes.  The router
    matches the oracle and repeats bit for bit (the split-K partial logits are
    summed in a fixed order)."""
    w = W.Workload(f"r{T}_{H}_{E}", T, H, E, k, 128, 128, mode, 2.826 if mode == "sigmoid" else 1.0,
                   0.0 if mode == "sigmoid" else 1e-8, True, "normal" if mode == "sigmoid" else "none",
                   0.1 if mode == "sigmoid" else 0.0, 21)
    inp, dl = _router_only(w)
    _check_route(w, inp, dl)
    a_idx, a_w, a_lg = dl.route()
    b_idx, b_w, b_lg = dl.route()
    torch.cuda.synchronize()
    assert torch.equal(a_idx, b_idx) and torch.equal(a_w, b_w) and torch.equal(a_lg, b_lg)


@pytest.mark.parametrize("name,T", [("prefill", 4096), ("zipf", 16384), ("image", 8192), ("prefill_u", 4096)])
def test_route_parity_full_size(name, T):
    """Router at the full workload sizes, every row (the oracle logits are one fp64 GEMM)."""
    w = W.WORKLOADS[name]
    hidden, router_w, bias = W.router_inputs(w)
    inp = {"hidden": hidden, "router_w": router_w, "bias": bias}
    dl = type("R", (), {})()
    dl.d = dims_of(w)
    dl.hidden, dl.router_w, dl.bias = bf16_dev(hidden), f32_dev(router_w), f32_dev(bias)
    dl.ws = moe.alloc_workspace(dl.d)
    dl.route = lambda: DeviceLayer.route(dl)
    gi, ref, ties = _check_route(w, inp, dl)
    assert moe.moe_ws_read_error(dl.ws) == 0
    print(f"{name}: near-tie rows where the GPU chose differently: {len(ties)}; "
          f"rows with margin < 1e-5: {int((ref['margin'] < NEAR_TIE).sum())}")


# ------------------------------------------------------------------ permutation

def _check_permute(w, topk):
    d = dims_of(w)
    dl = type("P", (), {})()
    dl.d = d
    dl.ws = moe.alloc_workspace(d)
    counts, offsets, perm, inv = DeviceLayer.permute(dl, i32_dev(topk))
    torch.cuda.synchronize()
    rc, ro = oracle.histogram_offsets(topk, w.E)
    rp, ri = oracle.permutation(topk, w.E)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(perm.cpu().numpy(), rp)
    assert np.array_equal(inv.cpu().numpy(), ri)
    assert moe.moe_ws_read_error(dl.ws) == 0


@pytest.mark.parametrize("w", [W.WORKLOADS["tiny"], MID, WIDE, DENSE, W.WORKLOADS["decode"], W.WORKLOADS["prefill"],
                               W.WORKLOADS["zipf"]], ids=["tiny", "mid", "wide", "dense", "decode", "prefill", "zipf"])
def test_permute_bit_exact(w):
    _check_permute(w, W.synthetic_topk(w))


def test_permute_skewed_and_empty_experts():
    """Expert 5 takes every token, expert 7 half of them, several experts none."""
    w = W.WORKLOADS["prefill"].with_(T=3001)
    topk = W.synthetic_topk(w) % 40          # only experts 0..39 can appear (plus 5 / 7 below)
    topk[:, 0] = 5
    topk[: w.T // 2, 1] = 7
    fixed = np.stack([_dedup(r, w.E) for r in topk])
    counts, _ = oracle.histogram_offsets(fixed, w.E)
    assert counts[5] == w.T and (counts == 0).sum() > 100
    _check_permute(w, fixed)


def _dedup(row, E):
    seen, out = set(), []
    for e in row.tolist():
        while e in seen:
            e = (e + 1) % E
        seen.add(e)
        out.append(e)
    return np.array(out, dtype=np.int32)


@pytest.mark.parametrize("T", [1024, 1025, 2047])
def test_permute_one_cta_many_cta_boundary(T):
    """S = T*8 around the switch from one CTA (S <= 8192) to 1024-slot parts, with a
    ragged last part: both paths give the oracle's stable permutation."""
    w = W.WORKLOADS["prefill"].with_(T=T)
    _check_permute(w, W.synthetic_topk(w))


def test_permute_many_cta_repeated_on_one_workspace():
    """The part counter in the workspace header is left zero: a second call on the
    same workspace (other indices) is exact too."""
    w = W.WORKLOADS["prefill"].with_(T=3000)
    d = dims_of(w)
    dl = type("P", (), {})()
    dl.d, dl.ws = d, moe.alloc_workspace(d)
    for shift in (0, 17):
        topk = np.stack([_dedup(r, w.E) for r in (W.synthetic_topk(w) + shift) % w.E])
        counts, offsets, perm, inv = DeviceLayer.permute(dl, i32_dev(topk))
        rp, ri = oracle.permutation(topk, w.E)
        assert np.array_equal(perm.cpu().numpy(), rp) and np.array_equal(inv.cpu().numpy(), ri)
        assert np.array_equal(offsets.cpu().numpy(), oracle.histogram_offsets(topk, w.E)[1])
    assert moe.moe_ws_read_error(dl.ws) == 0


def test_permute_many_cta_flags_out_of_range_index():
    w = W.WORKLOADS["prefill"].with_(T=2000)
    topk = W.synthetic_topk(w)
    topk[1500, 2] = -3
    d = dims_of(w)
    dl = type("P", (), {})()
    dl.d, dl.ws = d, moe.alloc_workspace(d)
    counts, offsets, perm, inv = DeviceLayer.permute(dl, i32_dev(topk))
    assert moe.moe_ws_read_error(dl.ws, clear=True) & moe.DEVERR_INDEX
    assert int(offsets[-1]) == w.S
    assert sorted(perm.cpu().numpy().tolist()) == list(range(w.S))


def test_permute_flags_out_of_range_index():
    w = W.WORKLOADS["tiny"]
    topk = W.synthetic_topk(w)
    topk[3, 1] = w.E + 7  # clamped on the device and reported
    d = dims_of(w)
    dl = type("P", (), {})()
    dl.d, dl.ws = d, moe.alloc_workspace(d)
    counts, offsets, perm, inv = DeviceLayer.permute(dl, i32_dev(topk))
    bits = moe.moe_ws_read_error(dl.ws, clear=True)
    assert bits & moe.DEVERR_INDEX
    assert int(offsets[-1]) == w.S
    assert sorted(perm.cpu().numpy().tolist()) == list(range(w.S))
    assert moe.moe_ws_read_error(dl.ws) == 0


# ------------------------------------------------------------------ expert FFN

@pytest.mark.parametrize("w", SMALL, ids=SMALL_IDS)
def test_expert_ffn_parity(w):
    """Given the oracle's own routing (perm/offsets), y_sorted and y_shared match the oracle."""
    inp = inputs_of(w)
    ref = oracle_layer(w, inp)
    dl = DeviceLayer(w, inp)
    y, z = dl.expert_ffn(i32_dev(ref["perm"]), i32_dev(ref["offsets"]))
    torch.cuda.synchronize()
    assert_layer_close(host_f64(y), ref["y_sorted"], f"{w.name} y_sorted")
    if w.has_shared:
        assert_layer_close(host_f64(z), ref["z"], f"{w.name} y_shared")
    assert moe.moe_ws_read_error(dl.ws) == 0


@pytest.mark.parametrize("T", [700, 512])
def test_expert_ffn_skewed_segments(T):
    """One expert holding every token (several chunks) and empty experts; these
    batches average at most 256 tokens per expert, so they run the 240-token tiles."""
    w = MID.with_(name="mid_skew", T=T)
    inp = W.layer_inputs(w)
    topk = np.zeros((w.T, 2), dtype=np.int32)
    topk[:, 0] = 3
    topk[:, 1] = np.where(np.arange(w.T) % 3 == 0, 6, 1)
    counts, offsets = oracle.histogram_offsets(topk, w.E)
    perm, inv = oracle.permutation(topk, w.E)
    y_ref = oracle.expert_outputs_sorted(inp["hidden"], perm, offsets, w.top_k, inp["w_gate"], inp["w_up"],
                                         inp["w_down"])
    dl = DeviceLayer(w, inp)
    y, z = dl.expert_ffn(i32_dev(perm), i32_dev(offsets))
    torch.cuda.synchronize()
    assert_layer_close(host_f64(y), y_ref, "skewed y_sorted")


def test_expert_ffn_widest_tiles():
    """T * k > 256 * E selects the 256-token tiles: one expert of two chunks of
    exactly 256 tokens, one of five chunks, one of three."""
    w = MID.with_(name="mid_wide_tiles", T=1040)
    assert w.T * w.top_k > 256 * w.E
    inp = W.layer_inputs(w)
    t = np.arange(w.T)
    topk = np.zeros((w.T, 2), dtype=np.int32)
    topk[:, 0] = 3
    topk[:, 1] = np.where(t < 512, 6, 1)
    counts, offsets = oracle.histogram_offsets(topk, w.E)
    assert counts[6] == 512 and counts[3] == 1040
    perm, inv = oracle.permutation(topk, w.E)
    y_ref = oracle.expert_outputs_sorted(inp["hidden"], perm, offsets, w.top_k, inp["w_gate"], inp["w_up"],
                                         inp["w_down"])
    z_ref = oracle.shared_expert(inp["hidden"], inp["ws_gate"], inp["ws_up"], inp["ws_down"])
    dl = DeviceLayer(w, inp)
    y, z = dl.expert_ffn(i32_dev(perm), i32_dev(offsets))
    torch.cuda.synchronize()
    assert_layer_close(host_f64(y), y_ref, "widest tiles y_sorted")
    assert_layer_close(host_f64(z), z_ref, "widest tiles y_shared")
    assert moe.moe_ws_read_error(dl.ws) == 0


def test_expert_ffn_odd_row_blocks_and_chunks():
    """Wide tiles with odd row-block counts (I = 384: three gate/up blocks; H = 768:
    three down blocks), an expert of three uneven chunks, one of ten tokens (a
    16-row activation tile), empty experts, and a one-block shared expert
    (I = 128) of three chunks."""
    w = W.Workload("pair_odd", 700, 768, 6, 2, 384, 128, "sigmoid", 2.826, 0.0, True, "normal", 0.1, 11)
    inp = W.layer_inputs(w)
    t = np.arange(w.T)
    topk = np.zeros((w.T, 2), dtype=np.int32)
    topk[:, 1] = np.where(t % 2 == 0, 4, np.where(t % 35 == 1, 2, 5))
    counts, offsets = oracle.histogram_offsets(topk, w.E)
    assert counts.tolist() == [700, 0, 10, 0, 350, 340]
    perm, inv = oracle.permutation(topk, w.E)
    y_ref = oracle.expert_outputs_sorted(inp["hidden"], perm, offsets, w.top_k, inp["w_gate"], inp["w_up"],
                                         inp["w_down"])
    z_ref = oracle.shared_expert(inp["hidden"], inp["ws_gate"], inp["ws_up"], inp["ws_down"])
    dl = DeviceLayer(w, inp)
    y, z = dl.expert_ffn(i32_dev(perm), i32_dev(offsets))
    torch.cuda.synchronize()
    assert_layer_close(host_f64(y), y_ref, "pair_odd y_sorted")
    assert_layer_close(host_f64(z), z_ref, "pair_odd y_shared")
    assert moe.moe_ws_read_error(dl.ws) == 0


def test_expert_ffn_decode_shape():
    """Hy3 decode shape (T = 8, 192 experts, I = 1536): N = 16 tiles, deep pipelines."""
    w = W.WORKLOADS["decode"]
    inp = inputs_of(w)
    ref = oracle_layer(w, inp)
    dl = DeviceLayer(w, inp)
    y, z = dl.expert_ffn(i32_dev(ref["perm"]), i32_dev(ref["offsets"]))
    torch.cuda.synchronize()
    assert_layer_close(host_f64(y), ref["y_sorted"], "decode y_sorted")
    assert_layer_close(host_f64(z), ref["z"], "decode y_shared")


# ------------------------------------------------------------------ stacked gate/up weights, routing given

@pytest.mark.parametrize("w", [W.WORKLOADS["tiny"], MID_SOFTMAX, NOSHARED, W.WORKLOADS["decode"]],
                         ids=["tiny", "mid_softmax", "noshared", "decode"])
def test_fused_moe_stacked_gate_up(w):
    """moe_fused_moe on [E, 2I, H] stacked gate/up weights (gate rows first)
    equals permute + expert FFN + combine on the separate tensors bit for bit,
    and matches the oracle's layer for the same routing."""
    inp = inputs_of(w)
    topk, wts = W.synthetic_topk(w, 3), W.synthetic_weights(w, 3)
    # renormalised as routing makes them (sum route_scale), which keeps |out| in
    # the range the layer tolerance is stated for
    wts = (wts / wts.sum(axis=1, keepdims=True) * w.route_scale).astype(np.float32)
    dl = DeviceLayer(w, inp)
    idx, wt = i32_dev(topk), f32_dev(wts)
    counts, offsets, perm, inv = dl.permute(idx)
    y, z = dl.expert_ffn(perm, offsets)
    staged = dl.combine(y, z, inv, wt)
    gu = torch.cat([dl.w_gate, dl.w_up], dim=1).contiguous()
    sgu = torch.cat([dl.ws_gate, dl.ws_up], dim=0).contiguous() if w.has_shared else None
    out = torch.empty_like(staged)
    moe.moe_fused_moe(dl.d, dl.hidden, idx, wt, gu, dl.w_down, sgu, dl.ws_down, out, dl.ws)
    out2 = moe.fused_moe(dl.hidden, idx, wt, gu, dl.w_down, ws_gate_up=sgu, ws_down=dl.ws_down)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), staged.view(torch.int16))
    assert torch.equal(out2.view(torch.int16), staged.view(torch.int16))
    assert moe.moe_ws_read_error(dl.ws) == 0
    _, offs_r = oracle.histogram_offsets(topk, w.E)
    perm_r, inv_r = oracle.permutation(topk, w.E)
    y_ref = oracle.expert_outputs_sorted(inp["hidden"], perm_r, offs_r, w.top_k, inp["w_gate"], inp["w_up"],
                                         inp["w_down"])
    z_ref = (oracle.shared_expert(inp["hidden"], inp["ws_gate"], inp["ws_up"], inp["ws_down"])
             if w.has_shared else None)
    ref = oracle.combine(y_ref, inv_r, wts.astype(np.float64), z_ref)
    assert_layer_close(host_f64(out), ref, f"{w.name} fused_moe")


# ------------------------------------------------------------------ combine

@pytest.mark.parametrize("w", [W.WORKLOADS["tiny"], MID, W.WORKLOADS["decode"], NOSHARED],
                         ids=["tiny", "mid", "decode", "noshared"])
def test_combine_parity(w):
    topk = W.synthetic_topk(w)
    perm, inv = oracle.permutation(topk, w.E)
    y = W.normal_bf16(w.seed, W.TID_AUX + 2, (w.S, w.H), 1.0)
    z = W.normal_bf16(w.seed, W.TID_AUX + 3, (w.T, w.H), 1.0) if w.has_shared else None
    wts = W.synthetic_weights(w)
    ref = oracle.combine(W.bf16_to_f64(y), inv, wts.astype(np.float64), None if z is None else W.bf16_to_f64(z))
    dl = type("C", (), {})()
    dl.d = dims_of(w)
    out = DeviceLayer.combine(dl, bf16_dev(y), None if z is None else bf16_dev(z), i32_dev(inv), f32_dev(wts))
    got = host_f64(out)
    # fp32 accumulation then one bf16 rounding: within half a bf16 ulp (<= 2^-8 |ref|)
    assert (np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-6).all()


# ------------------------------------------------------------------ whole layer

def _check_layer_rows(w, inp, got_rows, rows, gpu_idx_rows):
    """Compare sampled output rows with the oracle on those tokens; near-tie rows
    are compared with the oracle's output for the valid selection the GPU made."""
    hidden_rows = inp["hidden"][rows]
    ref = oracle_layer(w, inp, hidden=hidden_rows)
    same, ties = check_selection(gpu_idx_rows, ref, w.top_k)
    expected = ref["out"].copy()
    for t in ties:
        g = sorted(gpu_idx_rows[t].tolist())
        alts = valid_alternatives(ref, t, w.top_k)
        assert g in alts
        r2 = oracle_layer(w, inp, hidden=hidden_rows[t:t + 1], topk_idx=np.array([g], dtype=np.int32))
        expected[t] = r2["out"][0]
    return assert_layer_close(got_rows, expected, f"{w.name} layer rows"), len(ties)


@pytest.mark.parametrize("w", SMALL + [SMALL32, W.WORKLOADS["decode"]], ids=SMALL_IDS + ["small32", "decode"])
def test_layer_parity(w):
    inp = inputs_of(w)
    dl = DeviceLayer(w, inp)
    out = dl.forward()
    idx, _, _ = dl.route()
    torch.cuda.synchronize()
    got = host_f64(out)
    rows = np.arange(w.T)
    _check_layer_rows(w, inp, got, rows, idx.cpu().numpy())
    assert moe.moe_ws_read_error(dl.ws) == 0


@pytest.mark.parametrize("w", [W.WORKLOADS["tiny"], MID, SMALL32, W.WORKLOADS["decode"]],
                         ids=["tiny", "mid", "small32", "decode"])
def test_layer_equals_stage_chain_and_is_deterministic(w):
    inp = inputs_of(w)
    dl = DeviceLayer(w, inp)
    out1 = dl.forward()
    idx, wts, _ = dl.route()
    counts, offsets, perm, inv = dl.permute(idx)
    y, z = dl.expert_ffn(perm, offsets)
    out2 = dl.combine(y, z, inv, wts)
    out3 = dl.forward()
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(out1.view(torch.int16), out3.view(torch.int16))


def test_empty_batch_is_a_noop():
    w = W.WORKLOADS["tiny"].with_(T=0)
    d = dims_of(w)
    ws = moe.alloc_workspace(d)
    e = torch.empty(0, device="cuda")
    counts = torch.full((w.E,), 7, dtype=torch.int32, device="cuda")
    offsets = torch.full((w.E + 1,), 7, dtype=torch.int32, device="cuda")
    moe.moe_permute(d, torch.empty((0, w.top_k), dtype=torch.int32, device="cuda"), counts, offsets,
                    torch.empty(0, dtype=torch.int32, device="cuda"), torch.empty(0, dtype=torch.int32, device="cuda"),
                    ws)
    torch.cuda.synchronize()
    assert int(counts.abs().sum()) == 0 and int(offsets.abs().sum()) == 0
    del e


def test_single_token():
    w = W.WORKLOADS["tiny"].with_(name="t1", T=1)
    inp = W.layer_inputs(w)
    dl = DeviceLayer(w, inp)
    out = dl.forward()
    idx, _, _ = dl.route()
    torch.cuda.synchronize()
    _check_layer_rows(w, inp, host_f64(out), np.arange(1), idx.cpu().numpy())


# ------------------------------------------------------------------ full sizes (sampled)

def _sample_rows(T, n=24, seed=11):
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(4, T - 4), size=min(n - 8, max(0, T - 8)), replace=False)
    return np.unique(np.concatenate([np.arange(4), mid, np.arange(T - 4, T)]))


@pytest.mark.parametrize("name", ["prefill", "prefill_u", "zipf", "image"])
def test_layer_full_size_sampled(name):
    w = W.WORKLOADS[name]
    inp = W.layer_inputs(w)
    dl = DeviceLayer(w, inp)
    out = dl.forward()
    idx, wts, _ = dl.route()
    counts, offsets, perm, inv = dl.permute(idx)
    torch.cuda.synchronize()
    # properties at full size
    c, o, p, iv = (x.cpu().numpy() for x in (counts, offsets, perm, inv))
    gi = idx.cpu().numpy()
    assert c.sum() == w.S and o[0] == 0 and o[-1] == w.S and (np.diff(o) == c).all()
    assert np.array_equal(np.sort(p), np.arange(w.S))
    assert np.array_equal(iv[p], np.arange(w.S))
    flat = gi.reshape(-1)
    seg = np.repeat(np.arange(w.E), c)
    assert np.array_equal(flat[p], seg)                       # every slot sits in its expert's segment
    assert all((np.diff(p[o[e]:o[e + 1]]) > 0).all() for e in range(w.E))  # ascending slot order
    rows = _sample_rows(w.T)
    got = host_f64(out)[rows]
    (r, m), nties = _check_layer_rows(w, inp, got, rows, gi[rows])
    print(f"{name}: sampled rows {len(rows)} rel_l2={r:.3e} max_abs={m:.3e} near-tie rows={nties}; "
          f"expert counts max={c.max()} min={c.min()} empty={(c == 0).sum()}")
    assert moe.moe_ws_read_error(dl.ws) == 0


@pytest.mark.parametrize("name", ["prefill", "zipf", "image"])
def test_full_size_whole_segments_and_shared(name):
    """At full size, element by element: the whole y_sorted segment of the
    largest, a median and the smallest non-empty expert (every chunk, the ragged
    last one included) and all of y_shared, against the oracle's expert FFN on
    the same token rows (the GPU's own routing, which the sampled-layer test and
    the permutation tests check separately)."""
    w = W.WORKLOADS[name]
    inp = W.layer_inputs(w)
    dl = DeviceLayer(w, inp)
    idx, _, _ = dl.route()
    counts, offsets, perm, inv = dl.permute(idx)
    y, z = dl.expert_ffn(perm, offsets)
    torch.cuda.synchronize()
    c, o, p = counts.cpu().numpy(), offsets.cpu().numpy(), perm.cpu().numpy()
    nz = np.nonzero(c)[0]
    by = nz[np.argsort(c[nz], kind="stable")]
    picks = sorted({int(by[-1]), int(by[len(by) // 2]), int(by[0])})
    x = inp["hidden"]
    for e in picks:
        lo, hi = int(o[e]), int(o[e + 1])
        tok = p[lo:hi] // w.top_k
        ref = oracle.swiglu(x[tok], inp["w_gate"][e], inp["w_up"][e], inp["w_down"][e])
        assert_layer_close(host_f64(y[lo:hi]), ref, f"{name} expert {e} ({hi - lo} tokens) y_sorted")
    ref_z = oracle.shared_expert(x, inp["ws_gate"], inp["ws_up"], inp["ws_down"])
    assert_layer_close(host_f64(z), ref_z, f"{name} y_shared")
    assert moe.moe_ws_read_error(dl.ws) == 0


def test_bounded_wait_times_out_and_context_survives():
    """A kernel wait that nothing completes gives up after its limit, records
    MOE_DEVERR_TIMEOUT, and the GPU keeps working: a layer forward afterwards
    still matches the oracle."""
    w = W.WORKLOADS["tiny"]
    d = dims_of(w)
    ws = moe.alloc_workspace(d)
    moe.moe_selftest_wait_timeout(ws, 20_000_000)  # 20 ms
    bits = moe.moe_ws_read_error(ws, clear=True)
    assert bits & moe.DEVERR_TIMEOUT
    assert moe.moe_ws_read_error(ws) == 0
    inp = inputs_of(w)
    dl = DeviceLayer(w, inp)
    out = dl.forward()
    idx, _, _ = dl.route()
    torch.cuda.synchronize()
    _check_layer_rows(w, inp, host_f64(out), np.arange(w.T), idx.cpu().numpy())
