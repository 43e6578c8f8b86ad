"""Pins for the oracle's microscaling (MX) reading (oracle/mx.py): the E2M1
element format from its bit fields, nearest-even encoding by exhaustive
search, the shared block exponent by an integer search, block-level
properties, and the MX SwiGLU expert and layer against independently written
index loops."""
import math

import numpy as np

import oracle
import oracle.mx as MX
import workloads as W
from test_oracle_pins import _bf16_torch, _tiny_layer_inputs

# E2M1 (OCP MX v1.0, FP4): 1 sign, 2 exponent bits (bias 1; 0 = subnormal with
# value m * 2^-1), 1 mantissa bit; no infinities or NaN; largest 6.


def _e2m1_decode(code):
    sign = -1.0 if code & 0x8 else 1.0
    e, m = (code >> 1) & 0x3, code & 0x1
    return sign * (m * 0.5 if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1))


def _e4m3_decode(code):
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 15 and m == 7:
        return math.nan
    return sign * (m / 8.0 * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7))


_DECODE = {"e4m3": _e4m3_decode, "e2m1": _e2m1_decode}
_NPOS = {"e4m3": 0x7F, "e2m1": 0x8}        # non-negative finite codes 0 .. n-1
_SIGN = {"e4m3": 0x80, "e2m1": 0x8}
_MAXV = {"e4m3": 448.0, "e2m1": 6.0}
_EMAX = {"e4m3": 8, "e2m1": 2}             # exponent of the largest power of two each holds


def _encode_brute(x, elem):
    """Nearest non-negative finite value to |x| by exhaustive search (a tie to
    the even code, clamped to the largest value), then the sign of x."""
    dec = _DECODE[elem]
    a = min(abs(x), _MAXV[elem])
    best = min(range(_NPOS[elem]), key=lambda c: (abs(dec(c) - a), c & 1, c))
    return best | (_SIGN[elem] if math.copysign(1.0, x) < 0 else 0)


def _shared_exp_brute(amax, elem):
    """The largest e with 2^e <= amax by stepping, minus emax, clamped; -127 for 0."""
    if amax == 0:
        return -127
    e = 0
    while 2.0 ** e > amax:
        e -= 1
    while 2.0 ** (e + 1) <= amax:
        e += 1
    return max(-127, min(127, e - _EMAX[elem]))


def _quantize_mx_brute(row, elem):
    """One row, block by block: shared exponent, then every element by search."""
    codes, exps = [], []
    for b0 in range(0, len(row), 32):
        blk = [float(v) for v in row[b0:b0 + 32]]
        s = _shared_exp_brute(max(abs(v) for v in blk), elem)
        exps.append(s + 127)
        codes += [_encode_brute(v / 2.0 ** s, elem) for v in blk]
    return codes, exps


def test_e2m1_values_and_nearest_even_encoding():
    assert [float(MX.e2m1_value(c)) for c in range(8)] == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert [float(MX.e2m1_value(c)) for c in range(8, 16)] == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    assert all(float(MX.e2m1_value(c)) == _e2m1_decode(c) for c in range(16))
    pos = MX.e2m1_value(np.arange(8))
    mids = (pos[:-1] + pos[1:]) / 2                        # exact ties: 0.25 .. 5
    rng = np.random.default_rng(3)
    vals = np.concatenate([pos, -pos, mids, -mids, rng.uniform(-8, 8, 4000), [6.5, -100.0, 0.0, -0.0]])
    got = MX.e2m1_encode(vals)
    want = np.array([_encode_brute(float(v), "e2m1") for v in vals], dtype=np.uint8)
    assert np.array_equal(got, want)
    # ties: 0.25 -> 0 (code 0, even), 0.75 -> 1 (code 2), 1.25 -> 1 (code 2), 1.75 -> 2 (code 4), 2.5 -> 2, 3.5 -> 4, 5 -> 4
    assert [int(c) for c in MX.e2m1_encode([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])] == [0, 2, 2, 4, 4, 6, 6]


def test_shared_exponent_by_integer_search():
    vals = [0.0, 1e-45, 1e-40, 2.0 ** -130, 2.0 ** -120, 1.0, 255.0, 256.0, 257.0, 448.0, 511.9, 512.0, 1e30, 3e38]
    vals += [math.ldexp(1.0, k) for k in range(-140, 128, 7)]
    vals += [math.nextafter(math.ldexp(1.0, k), 0.0) for k in range(-100, 100, 13)]
    for elem in ("e4m3", "e2m1"):
        got = MX.mx_scale_exponent(np.array(vals), elem)
        want = [_shared_exp_brute(v, elem) for v in vals]
        assert [int(g) for g in got] == want, elem


def test_quantize_mx_blocks():
    rng = np.random.default_rng(11)
    v = rng.standard_normal((3, 128)) * np.array([[1e-3], [1.0], [50.0]])
    v[0, 32:64] = 0.0                                      # an all-zero block
    v[1, 64:96] *= 2.0 ** 9 / np.abs(v[1, 64:96]).max()    # block maximum exactly 2^9
    v[2, 96:128] *= 500.0 / np.abs(v[2, 96:128]).max()     # block maximum 500: 500 / 2^(8-8) saturates
    for elem in ("e4m3", "e2m1"):
        codes, exps, _ = MX.quantize_mx(v, elem)
        for r in range(3):
            bc, be = _quantize_mx_brute(v[r], elem)
            assert [int(c) for c in codes[r]] == bc and [int(e) for e in exps[r]] == be, (elem, r)
        assert int(exps[0, 1]) == 0 and not codes[0, 32:64].any()
        dec = MX.element_value(codes, elem)
        top = float(2.0 ** _EMAX[elem])                    # a power-of-two block maximum lands on 2^emax
        assert np.abs(dec[1, 64:96]).max() == top and int(exps[1, 2]) == 9 - _EMAX[elem] + 127
        assert np.abs(dec[2, 96:128]).max() == _MAXV[elem]  # saturated
        # scaling one block by 2^5 moves only its exponent
        v2 = v.copy()
        v2[1, :32] *= 32.0
        c2, e2, _ = MX.quantize_mx(v2, elem)
        assert np.array_equal(c2, codes) and int(e2[1, 0]) == int(exps[1, 0]) + 5
        assert np.array_equal(np.delete(e2, [4], axis=None), np.delete(exps, [4], axis=None))


def test_dequantize_mx_error_bound():
    rng = np.random.default_rng(12)
    v = rng.standard_normal((8, 256)) * 10.0 ** rng.uniform(-3, 3, (8, 1))
    for elem, rel, half_sub in (("e4m3", 2.0 ** -4, 2.0 ** -10), ("e2m1", 2.0 ** -2, 0.25)):
        codes, exps, _ = MX.quantize_mx(v, elem)
        deq = MX.dequantize_mx(codes, exps, elem)
        X = np.repeat(np.ldexp(1.0, exps.astype(np.int64) - 127), 32, axis=1)
        inside = np.abs(v) / X <= _MAXV[elem]
        err = np.abs(deq - v)
        bound = np.maximum(np.abs(v) * rel, X * half_sub)
        assert (err[inside] <= bound[inside] * (1 + 1e-12)).all(), elem
        assert np.array_equal(np.abs(deq[~inside]), X[~inside] * _MAXV[elem])


def _swiglu_mx_loops(x_row, g, u, d, a_elem):
    """One token through one MX SwiGLU expert with explicit index loops."""
    xq, xe = _quantize_mx_brute(x_row, a_elem)
    (gq, ge, gel), (uq, ue, uel), (dq, de, dl) = g, u, d
    I, H = gq.shape

    def dot(aq, ae, ael, wq, we, wel, n):
        return sum(_DECODE[ael](int(aq[h])) * 2.0 ** (int(ae[h // 32]) - 127) *
                   _DECODE[wel](int(wq[h])) * 2.0 ** (int(we[h // 32]) - 127) for h in range(n))

    a = []
    for i in range(I):
        gi = dot(xq, xe, a_elem, gq[i], ge[i], gel, H)
        ui = dot(xq, xe, a_elem, uq[i], ue[i], uel, H)
        a.append(gi / (1.0 + math.exp(-gi)) * ui)
    aq, ae = _quantize_mx_brute(_bf16_torch(np.array(a)), a_elem)
    return np.array([dot(aq, ae, a_elem, dq[o], de[o], dl, I) for o in range(dq.shape[0])])


def _mx_tiny(seed, T, H, E, I, Is, routed="e2m1", shared="e4m3"):
    x, wr, b, wg, wu, wd, sg, su, sd = _tiny_layer_inputs(seed, T, H, E, I, Is)
    experts = MX.quantize_experts_mx(wg, wu, wd, routed)
    shared_w = MX.quantize_experts_mx(sg, su, sd, shared)
    return x, wr, b, experts, shared_w, (wg, wu, wd, sg, su, sd)


def test_mx_swiglu_matches_index_loops():
    x, _, _, experts, shared, _ = _mx_tiny(51, 3, 64, 2, 32, 32)
    f = W.bf16_to_f64
    xq = MX.quantize_mx(f(x), "e4m3")
    (gq, ge, gel), (uq, ue, uel), (dq, de, dl) = experts
    pick = lambda a, e: (a[0][e], a[1][e], a[2])
    got = MX.swiglu_mx(xq, pick(experts[0], 1), pick(experts[1], 1), pick(experts[2], 1))
    got_s = MX.swiglu_mx(xq, *shared)
    for t in range(x.shape[0]):
        ref = _swiglu_mx_loops(f(x)[t], pick(experts[0], 1), pick(experts[1], 1), pick(experts[2], 1), "e4m3")
        np.testing.assert_allclose(got[t], ref, rtol=1e-12, atol=1e-13)
        ref_s = _swiglu_mx_loops(f(x)[t], *shared, "e4m3")
        np.testing.assert_allclose(got_s[t], ref_s, rtol=1e-12, atol=1e-13)


def test_mx_layer_matches_per_token_brute_force():
    T, H, E, k, I, Is = 4, 64, 4, 2, 32, 32
    x, wr, b, experts, shared, raw = _mx_tiny(52, T, H, E, I, Is)
    r = MX.layer_forward_mx(x, wr, b, experts, shared, top_k=k, route_scale=2.826)
    ref_route = oracle.layer_forward(x, wr, b, *raw, top_k=k)
    assert np.array_equal(r["idx"], ref_route["idx"]) and np.array_equal(r["w"], ref_route["w"])
    f = W.bf16_to_f64
    pick = lambda a, e: (a[0][e], a[1][e], a[2])
    for t in range(T):
        out = _swiglu_mx_loops(f(x)[t], *shared, "e4m3")
        for j, e in enumerate(r["idx"][t]):
            out = out + r["w"][t, j] * _swiglu_mx_loops(f(x)[t], pick(experts[0], e), pick(experts[1], e),
                                                        pick(experts[2], e), "e4m3")
        np.testing.assert_allclose(r["out"][t], out, rtol=1e-11, atol=1e-12)


def test_mx_layer_noise_against_the_bf16_layer():
    """Quantisation noise only: MXFP8 keeps 3 mantissa bits, MXFP4 one, so the
    all-MXFP8 layer stays within a few percent of the exact layer on the bf16
    weights and the hybrid (MXFP4 routed weights) within a few tens of percent,
    the MXFP8 one always the closer."""
    T, H, E, k, I, Is = 24, 64, 6, 2, 32, 32
    x, wr, b, _, _, raw = _mx_tiny(53, T, H, E, I, Is)
    exact = oracle.layer_forward(x, wr, b, *raw, top_k=k)["out"]
    rel = {}
    for routed in ("e4m3", "e2m1"):
        experts = MX.quantize_experts_mx(*raw[:3], routed)
        shared = MX.quantize_experts_mx(*raw[3:], "e4m3")
        out = MX.layer_forward_mx(x, wr, b, experts, shared, top_k=k)["out"]
        rel[routed] = np.linalg.norm(out - exact) / np.linalg.norm(exact)
    assert 1e-4 < rel["e4m3"] < 0.08, rel
    assert rel["e4m3"] < rel["e2m1"] < 0.4, rel
