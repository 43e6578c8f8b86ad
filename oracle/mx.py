"""Microscaling (MX) block formats for the oracle: MXFP8 (E4M3 elements) and
MXFP4 (E2M1 elements), and the MoE layer with MX experts.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing on the product
path may import, call or execute it.

The Ascend deployment article (section 8.2) replaces FP8 with MXFP8 in the
Linear modules -- W8A8 for the attention projections and the shared expert --
and gives the routed experts MXFP4 weights with MXFP8 activations (W4A8), the
activations quantised dynamically; it fixes no further detail.  Reading: the
OCP Microscaling formats (MX specification v1.0).  Blocks of 32 consecutive
values along the reduction axis share one power-of-two scale
X = 2^(floor(log2 max|v|) - emax), kept as a biased 8-bit exponent (UE8M0, bias
127; the unbiased exponent clamped to [-127, 127]).  emax is the exponent of the
element format's largest power of two: 8 for E4M3 (256), 2 for E2M1 (4).  Each
element is v / X (exact: X is a power of two) rounded to the nearest element
value, ties to the even code, magnitudes past the largest finite value (448
for E4M3, 6 for E2M1) saturated to it.  An all-zero block gets X = 2^-127.
"""
from __future__ import annotations

import numpy as np

from .moe import (bf16_round, combine, e4m3_encode, e4m3_value, histogram_offsets, permutation, route_sigmoid,
                  route_softmax, router_logits, routing_weights_for, silu, widen_bf16)

MX_BLOCK = 32
MX_EMAX = {"e4m3": 8, "e2m1": 2}


def e2m1_value(code) -> np.ndarray:
    """Real value of E2M1 codes (4 bits: sign, 2 exponent bits with bias 1 and
    0 = subnormal, 1 mantissa bit): 0, 0.5, 1, 1.5, 2, 3, 4, 6 and negatives."""
    c = np.asarray(code, dtype=np.int64)
    sign = np.where(c & 0x8, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = c & 0x1
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * 2.0 ** (e - 1.0))
    return sign * mag


def e2m1_encode(v) -> np.ndarray:
    """Nearest E2M1 code (ties to the even code), magnitudes past 6 saturated to 6."""
    v = np.asarray(v, dtype=np.float64)
    pos = e2m1_value(np.arange(8))             # 0 .. 6, increasing, codes 0x0..0x7
    a = np.minimum(np.abs(v), 6.0)
    hi = np.clip(np.searchsorted(pos, a, side="left"), 0, 7)
    lo = np.maximum(hi - 1, 0)
    dlo, dhi = a - pos[lo], pos[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.int64)
    code = np.where(np.signbit(v), code | 0x8, code)
    return code.astype(np.uint8)


def element_value(code, elem: str) -> np.ndarray:
    return e4m3_value(code) if elem == "e4m3" else e2m1_value(code)


def element_encode(v, elem: str) -> np.ndarray:
    return e4m3_encode(v) if elem == "e4m3" else e2m1_encode(v)


def mx_scale_exponent(amax, elem: str) -> np.ndarray:
    """Unbiased shared exponent of blocks whose largest magnitude is amax:
    floor(log2 amax) - emax, clamped to [-127, 127]; -127 for an all-zero block."""
    a = np.asarray(amax, dtype=np.float64)
    _, e2 = np.frexp(np.where(a > 0, a, 1.0))  # a = f * 2^e2, f in [0.5, 1): floor(log2 a) = e2 - 1
    shared = (e2 - 1) - MX_EMAX[elem]
    return np.where(a > 0, np.clip(shared, -127, 127), -127).astype(np.int64)


def quantize_mx(v, elem: str):
    """MX quantisation along the last axis (a multiple of 32): returns (codes
    uint8 [..., n], biased scale exponents uint8 [..., n / 32], elem)."""
    v = np.asarray(v, dtype=np.float64)
    n = v.shape[-1]
    if n % MX_BLOCK:
        raise ValueError("the blocked axis must be a multiple of 32")
    blocks = v.reshape(v.shape[:-1] + (n // MX_BLOCK, MX_BLOCK))
    shared = mx_scale_exponent(np.abs(blocks).max(axis=-1), elem)
    codes = element_encode(blocks / np.ldexp(1.0, shared)[..., None], elem)
    return codes.reshape(v.shape), (shared + 127).astype(np.uint8), elem


def dequantize_mx(codes, exps, elem: str) -> np.ndarray:
    """The values an MX tensor stands for: value(code) * 2^(exp - 127), exactly."""
    c = np.asarray(codes)
    n = c.shape[-1]
    vals = element_value(c, elem).reshape(c.shape[:-1] + (n // MX_BLOCK, MX_BLOCK))
    scale = np.ldexp(1.0, np.asarray(exps, dtype=np.int64) - 127)
    return (vals * scale[..., None]).reshape(c.shape)


def mx_linear(x, w) -> np.ndarray:
    """out[t, o] = sum_h x[t, h] * w[o, h] for an input and a weight that are
    both MX tensors (codes, exponents, element format) blocked along h: each
    block's code products times the two block scales, summed over the blocks."""
    return dequantize_mx(*x) @ dequantize_mx(*w).T


def swiglu_mx(x, g, u, d, a_elem: str = "e4m3") -> np.ndarray:
    """One SwiGLU expert with MX weights g, u, d: gate and up from the MX input
    rows x, the activation SiLU(gate) * up stored as bf16 and MX-quantised along
    its row (the down GEMM's reduction axis), then the down projection."""
    gate = mx_linear(x, g)
    up = mx_linear(x, u)
    a = bf16_round(silu(gate) * up)
    return mx_linear(quantize_mx(a, a_elem), d)


def quantize_experts_mx(w_gate, w_up, w_down, elem: str):
    """Stacked expert weights [E, rows, cols] (bf16 bits or floats), each row MX
    quantised along its input axis."""
    f = lambda a: quantize_mx(widen_bf16(a) if np.asarray(a).dtype == np.uint16 else a, elem)
    return f(w_gate), f(w_up), f(w_down)


def layer_forward_mx(hidden, router_w, bias, experts, shared, *, top_k: int, score_mode: str = "sigmoid",
                     route_scale: float = 2.826, renorm_eps: float = 0.0, a_elem: str = "e4m3", topk_idx=None):
    """The layer with MX experts.  `experts` = (gate, up, down), each an MX
    tensor from quantize_mx along the input axis (codes [E, rows, cols],
    exponents [E, rows, cols / 32], element format); `shared` likewise (or None).
    The Ascend article's hybrid is MXFP4 (e2m1) routed weights, MXFP8 (e4m3)
    shared weights and MXFP8 activations.  Routing as in layer_forward (fp32
    router, unquantised); each token's hidden row is quantised once (a_elem)."""
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
    _, offsets = histogram_offsets(idx, E)
    perm, inv = permutation(idx, E)
    hq, he, _ = quantize_mx(widen_bf16(hidden), a_elem)
    (gq, ge, gel), (uq, ue, uel), (dq, de, dl) = experts
    tok = np.asarray(perm, dtype=np.int64) // top_k
    y = np.zeros((tok.size, np.asarray(hidden).shape[1]), dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            t = tok[lo:hi]
            y[lo:hi] = swiglu_mx((hq[t], he[t], a_elem), (gq[e], ge[e], gel), (uq[e], ue[e], uel),
                                 (dq[e], de[e], dl), a_elem)
    z = swiglu_mx((hq, he, a_elem), *shared, a_elem) if shared is not None else None
    out = combine(y, inv, w, z)
    return {"idx": idx, "w": w, "perm": perm, "inv": inv, "offsets": offsets, "y_sorted": y, "z": z, "out": out}
