"""fp64 oracle of one MoE FFN layer forward (test infrastructure only; see the
package docstring for the sources and the readings)."""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# storage conversions
# ---------------------------------------------------------------------------


def widen_bf16(a) -> np.ndarray:
    """bf16 tensors arrive as uint16 bit patterns; widen them exactly to float64.
    Float arrays are widened with astype (exact for fp32)."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def bf16_round(v) -> np.ndarray:
    """Round fp32-representable values to the nearest bf16, ties to even
    (8 significant bits).  Returns float64 holding the bf16 values."""
    v32 = np.asarray(v, dtype=np.float32)
    u = v32.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# a1  router GEMM
# ---------------------------------------------------------------------------


def router_logits(x, router_w) -> np.ndarray:
    """logits[t, e] = sum_h x[t, h] * Wr[e, h] with the fp32 router weight taken
    exactly (HunyuanTopKGate: Linear(H -> E, bias=False, float32) applied to the
    hidden state cast to float; hy3 README keeps the router in F32).  This is the
    plain definition the two-BF16 split approximates."""
    return widen_bf16(x) @ widen_bf16(router_w).T


def split_router_weight(router_w):
    """The two-BF16 reconstruction of the fp32 router weight (Hy3 Preview case,
    section 2): W ~ W_high + scale * W_low with scale = 1/256.  Reading:
    W_high = bf16_RNE(W), W_low = bf16_RNE((W - W_high) * 256).  W - W_high and
    the product by 256 are exact in fp32."""
    w = np.asarray(router_w, dtype=np.float32)
    w_high = bf16_round(w)
    resid = (w.astype(np.float64) - w_high) * 256.0
    w_low = bf16_round(resid.astype(np.float32))
    return w_high, w_low


def router_logits_split(x, w_high, w_low) -> np.ndarray:
    """What two BF16 GEMMs with two accumulators and one FFMA epilogue compute,
    without accumulation rounding: acc_hi + acc_lo * (1/256)."""
    xd = widen_bf16(x)
    return xd @ w_high.T + (xd @ w_low.T) * (1.0 / 256.0)


# ---------------------------------------------------------------------------
# a2  scoring, top-k, renormalisation
# ---------------------------------------------------------------------------


def sigmoid(z):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-np.asarray(z, dtype=np.float64)))


def silu(g):
    """SiLU(g) = g * sigmoid(g) = g / (1 + exp(-g))."""
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def topk_desc(keys, k: int):
    """Indices of the k largest keys per row, in descending key order; equal
    keys go to the lower expert index.  Full sort (brute force).  Also returns
    margin = key_(k) - key_(k+1) (+inf when k == E)."""
    keys = np.asarray(keys, dtype=np.float64)
    order = np.argsort(-keys, axis=1, kind="stable")
    idx = order[:, :k]
    kth = np.take_along_axis(keys, order[:, k - 1:k], axis=1)[:, 0]
    if k < keys.shape[1]:
        nxt = np.take_along_axis(keys, order[:, k:k + 1], axis=1)[:, 0]
        margin = kth - nxt
    else:
        margin = np.full(keys.shape[0], np.inf)
    return idx.astype(np.int32), margin


def renormalize(sel, eps: float) -> np.ndarray:
    """sel / clamp(sum(sel), min=eps) per row (easy_topk); eps = 0 is the plain
    renormalisation to sum 1 of the sigmoid rule."""
    sel = np.asarray(sel, dtype=np.float64)
    tot = sel.sum(axis=1, keepdims=True)
    return sel / np.maximum(tot, eps)


def route_sigmoid(logits, bias, k: int, route_scale: float):
    """hy3 README, Model facts, MoE routing: s = sigmoid(logits); the top-k is
    chosen on s + expert_bias; the weights are the unbiased s of the chosen
    experts renormalised to sum 1, then multiplied by route_scale (2.826)."""
    s = sigmoid(logits)
    keys = s + (0.0 if bias is None else widen_bf16(bias)[None, :])
    idx, margin = topk_desc(keys, k)
    s_sel = np.take_along_axis(s, idx, axis=1)
    w = renormalize(s_sel, 0.0) * route_scale
    return {"idx": idx, "w": w, "margin": margin, "keys": keys, "scores": s}


def route_softmax(logits, k: int, eps: float = 1e-8):
    """HunyuanTopKGate easy_topk: gates = softmax(logits, dim=experts); top-k of
    gates; weights = top-k gates / clamp(sum, min=eps)."""
    lg = np.asarray(logits, dtype=np.float64)
    ex = np.exp(lg - lg.max(axis=1, keepdims=True))
    p = ex / ex.sum(axis=1, keepdims=True)
    idx, margin = topk_desc(p, k)
    w = renormalize(np.take_along_axis(p, idx, axis=1), eps)
    return {"idx": idx, "w": w, "margin": margin, "keys": p, "scores": p}


def routing_weights_for(scores, idx, score_mode: str, route_scale: float, eps: float):
    """Combine weights for a given (valid) selection, from the oracle's own scores:
    sigmoid rule -> s_sel / sum * route_scale; softmax rule -> p_sel / clamp(sum, eps)."""
    sel = np.take_along_axis(np.asarray(scores, dtype=np.float64), np.asarray(idx, dtype=np.int64), axis=1)
    if score_mode == "sigmoid":
        return renormalize(sel, 0.0) * route_scale
    return renormalize(sel, eps)


def near_tie_alternatives(keys, k: int, tol: float):
    """For each row, the experts that any valid top-k must hold (key above the
    k-th key by more than tol) and the experts that may fill the remaining
    places (key within tol of the k-th key).  A selection G of a row is valid
    iff mandatory <= G <= mandatory | candidates and |G| = k."""
    keys = np.asarray(keys, dtype=np.float64)
    kth = -np.sort(-keys, axis=1)[:, k - 1:k]
    mandatory = keys > kth + tol
    candidate = np.abs(keys - kth) <= tol
    return mandatory, candidate


# ---------------------------------------------------------------------------
# a3, a4  histogram, offsets, permutation
# ---------------------------------------------------------------------------


def histogram_offsets(topk_idx, E: int):
    """cnt[e] = number of (t, j) with topk_idx[t, j] == e; offsets = exclusive
    prefix sum of cnt, length E + 1 (one contiguous range per expert)."""
    flat = np.asarray(topk_idx, dtype=np.int64).reshape(-1)
    counts = np.bincount(flat, minlength=E)[:E].astype(np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    return counts, offsets


def permutation(topk_idx, E: int):
    """Following the eager path of the HunyuanImage post: flatten topk_idx (slot
    t*k + j), and for each expert e in order take the slots routed to it
    (flat == e) in ascending slot order.  perm[p] = slot at sorted position p;
    inv[slot] = p."""
    flat = np.asarray(topk_idx, dtype=np.int64).reshape(-1)
    S = flat.size
    perm = np.empty(S, dtype=np.int32)
    pos = 0
    for e in range(E):
        slots = np.nonzero(flat == e)[0]
        perm[pos:pos + slots.size] = slots
        pos += slots.size
    assert pos == S, "routing index outside [0, E)"
    inv = np.empty(S, dtype=np.int32)
    inv[perm] = np.arange(S, dtype=np.int32)
    return perm, inv


# ---------------------------------------------------------------------------
# a5-a8  expert FFNs
# ---------------------------------------------------------------------------


def swiglu(x, w_gate, w_up, w_down) -> np.ndarray:
    """SwiGLU expert: down(SiLU(gate(x)) * up(x)) with nn.Linear [out, in] weights."""
    xd = widen_bf16(x)
    g = xd @ widen_bf16(w_gate).T
    u = xd @ widen_bf16(w_up).T
    a = silu(g) * u
    return a @ widen_bf16(w_down).T


def expert_outputs_sorted(hidden, perm, offsets, top_k: int, w_gate, w_up, w_down) -> np.ndarray:
    """y_sorted[p] = FFN_e(x[perm[p] // k]) for p in expert e's range: the eager
    per-expert loop, with rows already grouped by expert."""
    x = widen_bf16(hidden)
    perm = np.asarray(perm, dtype=np.int64)
    S = perm.size
    y = np.zeros((S, x.shape[1]), dtype=np.float64)
    E = len(offsets) - 1
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        tokens = perm[lo:hi] // top_k
        y[lo:hi] = swiglu(x[tokens], w_gate[e], w_up[e], w_down[e])
    return y


def shared_expert(hidden, ws_gate, ws_up, ws_down) -> np.ndarray:
    """Shared MLP: the same SwiGLU on every token, no router, no gate, no scale."""
    return swiglu(hidden, ws_gate, ws_up, ws_down)


# ---------------------------------------------------------------------------
# a9  combine
# ---------------------------------------------------------------------------


def combine(y_sorted, inv, topk_w, z=None) -> np.ndarray:
    """out[t] = sum_j w[t, j] * y_sorted[inv[t*k + j]] (+ z[t]): reshape the
    expert outputs to [T, k, H], weight them, sum over k, add the shared branch."""
    w = np.asarray(topk_w, dtype=np.float64)
    T, k = w.shape
    y = np.asarray(y_sorted, dtype=np.float64)
    inv = np.asarray(inv, dtype=np.int64).reshape(T, k)
    out = (y[inv] * w[:, :, None]).sum(axis=1)
    if z is not None:
        out = out + np.asarray(z, dtype=np.float64)
    return out


# ---------------------------------------------------------------------------
# FP8 (E4M3) expert weights with one scale per output row
# ---------------------------------------------------------------------------
# The Hy3 case lists W8A8 among its quantised deployments and quantises inside
# the FusedMoE chain; the pages fix neither the format nor the scaling.  The
# reading here (weight-only): every expert matrix is stored as OCP FP8 E4M3
# codes (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 is
# subnormal; S.1111.111 is NaN, so the largest finite magnitude is 448) with one
# fp32 scale per output row, scale = max|row| / 448 (1 for an all-zero row);
# the layer uses value(code) * scale, exactly, in place of each bf16 weight
# (the scale multiplies the matrix product of a row, so no rounding of the
# product of code and scale enters).


def e4m3_value(code) -> np.ndarray:
    """Real value of E4M3 codes (uint8), NaN for the two NaN codes."""
    c = np.asarray(code, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(v) -> np.ndarray:
    """Nearest E4M3 code (ties to the even code), magnitudes past 448 saturated
    to 448, NaN to the NaN code.  v is taken as float64 (the callers pass fp32
    values)."""
    v = np.asarray(v, dtype=np.float64)
    pos = e4m3_value(np.arange(0x7F))          # 0 .. 448, increasing, codes 0x00..0x7E
    a = np.minimum(np.abs(v), 448.0)
    hi = np.clip(np.searchsorted(pos, a, side="left"), 0, 0x7E)
    lo = np.maximum(hi - 1, 0)
    dlo, dhi = a - pos[lo], pos[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.int64)
    code = np.where(np.signbit(v), code | 0x80, code)
    code = np.where(np.isnan(v), 0x7F, code)
    return code.astype(np.uint8)


def quantize_rows_e4m3(w):
    """Per output row (last axis = input features): scale = fp32(max|w|) / 448 in
    fp32 (1 if the row is zero), code = e4m3_encode(fp32(w) / scale) with the
    division in fp32.  Returns (codes uint8, scales float32)."""
    w32 = widen_bf16(w).astype(np.float32)
    amax = np.abs(w32).max(axis=-1)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    q = e4m3_encode((w32 / scale[..., None]).astype(np.float32))
    return q, scale


def dequantize_rows_e4m3(q, scale) -> np.ndarray:
    """The weight a stored row stands for: value(code) * scale, exact in float64
    (at most 4 significant bits times 24)."""
    return e4m3_value(q) * np.asarray(scale, dtype=np.float64)[..., None]


# ---------------------------------------------------------------------------
# W8A8: FP8 (E4M3) weights and FP8 activations
# ---------------------------------------------------------------------------
# The Hy3 case's FusedMoE chain quantises the activations right before the down
# GEMM ("activation quantisation + Down GEMM") in its W8A8 deployments; the
# pages fix no format or granularity.  The reading here: the weights as above
# (E4M3 codes, one fp32 scale per output row), and every activation matrix that
# feeds a GEMM quantised the same way per row, dynamically from its own values:
# the hidden state per token before the gate/up GEMM, and the SiLU(gate) * up
# activation per routed slot (per token for the shared expert) before the down
# GEMM.  The activation the down GEMM quantises is the bf16 value the layer
# stores between the two GEMMs.  Products of two codes are exact, so each
# output element is (sum of code products) * row scale * column scale.  The
# router is not quantised (it stays in fp32).


def quantized_matmul(xq, xs, wq, ws) -> np.ndarray:
    """out[t, o] = sum_h value(xq[t, h]) * value(wq[o, h]) * xs[t] * ws[o]: an
    nn.Linear whose input rows and weight rows are both E4M3 codes with one
    scale per row."""
    acc = e4m3_value(xq) @ e4m3_value(wq).T
    return acc * np.asarray(xs, dtype=np.float64)[:, None] * np.asarray(ws, dtype=np.float64)[None, :]


def swiglu_w8a8(xq, xs, g, u, d) -> np.ndarray:
    """One SwiGLU expert, W8A8: gate and up from the quantised input rows, the
    activation a = SiLU(gate) * up stored as bf16 and quantised per row, then the
    down projection.  g, u, d are (codes, scales) pairs of the three weights."""
    gate = quantized_matmul(xq, xs, *g)
    up = quantized_matmul(xq, xs, *u)
    a = bf16_round(silu(gate) * up)
    aq, a_s = quantize_rows_e4m3(a)
    return quantized_matmul(aq, a_s, *d)


def layer_forward_w8a8(hidden, router_w, bias, experts, shared, *, top_k: int, score_mode: str = "sigmoid",
                       route_scale: float = 2.826, renorm_eps: float = 0.0, topk_idx=None):
    """The layer with W8A8 experts.  `experts` = (gate, up, down), each a
    (codes [E, rows, cols], scales [E, rows]) pair from quantize_rows_e4m3;
    `shared` likewise for the shared expert (or None).  Routing as in
    layer_forward (fp32 router, unquantised); each token's hidden row is
    quantised once and read through the route index by every expert it visits."""
    E = np.asarray(router_w).shape[0]
    logits = router_logits(hidden, router_w)
    if score_mode == "sigmoid":
        r = route_sigmoid(logits, bias, top_k, route_scale)
    elif score_mode == "softmax":
        r = route_softmax(logits, top_k, renorm_eps)
    else:
        raise ValueError(score_mode)
    idx, w = r["idx"], r["w"]
    if topk_idx is not None:
        idx = np.asarray(topk_idx, dtype=np.int32)
        w = routing_weights_for(r["scores"], idx, score_mode, route_scale, renorm_eps)
    counts, offsets = histogram_offsets(idx, E)
    perm, inv = permutation(idx, E)
    hq, hs = quantize_rows_e4m3(hidden)
    (gq, gs), (uq, us), (dq, ds) = experts
    tok = np.asarray(perm, dtype=np.int64) // top_k
    y = np.zeros((tok.size, np.asarray(hidden).shape[1]), dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            t = tok[lo:hi]
            y[lo:hi] = swiglu_w8a8(hq[t], hs[t], (gq[e], gs[e]), (uq[e], us[e]), (dq[e], ds[e]))
    z = swiglu_w8a8(hq, hs, *shared) if shared is not None else None
    out = combine(y, inv, w, z)
    return {"idx": idx, "w": w, "margin": r["margin"], "keys": r["keys"], "perm": perm, "inv": inv,
            "offsets": offsets, "y_sorted": y, "z": z, "out": out}


# ---------------------------------------------------------------------------
# whole layer
# ---------------------------------------------------------------------------


def layer_forward(hidden, router_w, bias, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, *,
                  top_k: int, score_mode: str = "sigmoid", route_scale: float = 2.826,
                  renorm_eps: float = 0.0, topk_idx=None):
    """One MoE FFN layer forward, every intermediate in float64.

    If ``topk_idx`` is given it replaces the oracle's own selection (it must be
    a valid selection, see near_tie_alternatives); the weights are then the
    oracle's own for that selection."""
    E = np.asarray(router_w).shape[0]
    logits = router_logits(hidden, router_w)
    if score_mode == "sigmoid":
        r = route_sigmoid(logits, bias, top_k, route_scale)
    elif score_mode == "softmax":
        r = route_softmax(logits, top_k, renorm_eps)
    else:
        raise ValueError(score_mode)
    idx, w = r["idx"], r["w"]
    if topk_idx is not None:
        idx = np.asarray(topk_idx, dtype=np.int32)
        w = routing_weights_for(r["scores"], idx, score_mode, route_scale, renorm_eps)
    counts, offsets = histogram_offsets(idx, E)
    perm, inv = permutation(idx, E)
    y = expert_outputs_sorted(hidden, perm, offsets, top_k, w_gate, w_up, w_down)
    z = shared_expert(hidden, ws_gate, ws_up, ws_down) if ws_gate is not None else None
    out = combine(y, inv, w, z)
    return {"logits": logits, "idx": idx, "w": w, "margin": r["margin"], "keys": r["keys"],
            "scores": r["scores"], "counts": counts, "offsets": offsets, "perm": perm, "inv": inv,
            "y_sorted": y, "z": z, "out": out}


def layer_rows(rows_hidden, router_w, bias, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, **kw):
    """The layer on a sample of tokens.  Every step is token-wise (routing per
    row, one FFN per token copy, combine per token), so the output rows of a
    sample equal the same rows of the full batch; only the sorted order differs."""
    return layer_forward(rows_hidden, router_w, bias, w_gate, w_up, w_down,
                         ws_gate, ws_up, ws_down, **kw)
