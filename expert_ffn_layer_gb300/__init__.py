"""Python binding of libmoe_gb300.so (include/moe.h): argument marshalling only.

Every step of the layer runs in the library's CUDA kernels; PyTorch is used
here for device memory and streams.  There is no fallback: if the library is
missing or a call fails, an exception is raised.

Function names follow the C ABI:

    moe_route, moe_permute, moe_expert_ffn (= moe_expert_gate_up + moe_expert_down),
    moe_combine, moe_layer_forward,
    moe_fused_moe (routing given, stacked [E, 2I, H] gate/up weights),
    moe_quantize_fp8_rows, moe_expert_ffn_fp8, moe_layer_forward_fp8 (FP8 E4M3
    expert weights, one scale per row; see Fp8Experts / quantize_fp8_experts),
    moe_workspace_bytes, moe_ws_init, moe_ws_read_error, moe_check_dims

Tensors are torch tensors on the current CUDA device: bf16 activations and
weights, fp32 router weight / bias / combine weights, int32 indices, a uint8
workspace of moe_workspace_bytes(d) bytes (see ``alloc_workspace``).
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

from .build import LIB as _LIB_PATH

MOE_OK = 0
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_TIMEOUT", 6: "MOE_ERR_DEVICE_INDEX"}
DEVERR_INDEX, DEVERR_TIMEOUT, DEVERR_OFFSETS = 0x1, 0x2, 0x4
SCORE_SIGMOID_BIAS, SCORE_SOFTMAX = 0, 1

EXPORTS = ("moe_status_string", "moe_check_dims", "moe_workspace_bytes", "moe_ws_init", "moe_ws_read_error",
           "moe_route", "moe_permute", "moe_expert_ffn", "moe_expert_gate_up", "moe_expert_down", "moe_combine",
           "moe_layer_forward", "moe_fused_moe", "moe_expert_ffn_noalloc", "moe_selftest_wait_timeout",
           "moe_selftest_silu", "moe_quantize_fp8_rows", "moe_expert_ffn_fp8", "moe_layer_forward_fp8",
           "moe_expert_ffn_w8a8", "moe_layer_forward_w8a8")


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)}")


class MoeDims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("E", ctypes.c_int), ("I", ctypes.c_int),
                ("I_shared", ctypes.c_int), ("top_k", ctypes.c_int), ("score_mode", ctypes.c_int),
                ("route_scale", ctypes.c_float), ("renorm_eps", ctypes.c_float), ("has_shared", ctypes.c_int)]

    def __repr__(self):
        return "MoeDims(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


class MoeFp8Experts(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("gate", "up", "down", "gate_scale", "up_scale", "down_scale",
                                                "s_gate", "s_up", "s_down", "s_gate_scale", "s_up_scale",
                                                "s_down_scale")]


_lib = None


def library_path() -> Path:
    return _LIB_PATH


def load() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not _LIB_PATH.exists():
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with expert_ffn_layer_gb300.build.build() "
                           "(or __graft_entry__.build()); there is no CPU fallback")
    lib = ctypes.CDLL(str(_LIB_PATH))
    P, C = ctypes.c_void_p, ctypes.c_size_t
    D = ctypes.POINTER(MoeDims)
    st = ctypes.c_int
    sig = {
        "moe_status_string": (ctypes.c_char_p, [st]),
        "moe_check_dims": (st, [D]),
        "moe_workspace_bytes": (C, [D]),
        "moe_ws_init": (st, [P, C, P]),
        "moe_ws_read_error": (st, [P, C, ctypes.c_int, P, ctypes.POINTER(ctypes.c_uint32)]),
        "moe_route": (st, [D, P, P, P, P, P, P, P, C, P]),
        "moe_permute": (st, [D, P, P, P, P, P, P, C, P]),
        "moe_expert_ffn": (st, [D, P, P, P, P, P, P, P, P, P, P, P, P, C, P]),
        "moe_expert_gate_up": (st, [D, P, P, P, P, P, P, P, P, C, P]),
        "moe_expert_down": (st, [D, P, P, P, P, P, P, C, P]),
        "moe_combine": (st, [D, P, P, P, P, P, P]),
        "moe_layer_forward": (st, [D, P, P, P, P, P, P, P, P, P, P, P, C, P]),
        "moe_fused_moe": (st, [D, P, P, P, P, P, P, P, P, P, C, P]),
        "moe_quantize_fp8_rows": (st, [P, ctypes.c_int64, ctypes.c_int, P, P, P]),
        "moe_expert_ffn_fp8": (st, [D, P, P, P, ctypes.POINTER(MoeFp8Experts), P, P, P, C, P]),
        "moe_layer_forward_fp8": (st, [D, P, P, P, ctypes.POINTER(MoeFp8Experts), P, P, C, P]),
        "moe_expert_ffn_w8a8": (st, [D, P, P, P, ctypes.POINTER(MoeFp8Experts), P, P, P, C, P]),
        "moe_layer_forward_w8a8": (st, [D, P, P, P, ctypes.POINTER(MoeFp8Experts), P, P, C, P]),
        "moe_selftest_wait_timeout": (st, [P, C, ctypes.c_ulonglong, P]),
        "moe_selftest_silu": (st, [P, P, P, ctypes.c_int64, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().moe_status_string(status).decode()


def dims(T: int, H: int, E: int, I: int, top_k: int, I_shared: int | None = None, score_mode: str = "sigmoid",
         route_scale: float = 2.826, renorm_eps: float = 0.0, has_shared: bool = True) -> MoeDims:
    mode = {"sigmoid": SCORE_SIGMOID_BIAS, "softmax": SCORE_SOFTMAX}[score_mode]
    return MoeDims(T, H, E, I, I if I_shared is None else I_shared, top_k, mode, route_scale, renorm_eps,
                   1 if has_shared else 0)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _check(t, dtype, shape, name):
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _call(fn: str, *args):
    rc = getattr(load(), fn)(*args)
    if rc != MOE_OK:
        raise MoeError(fn, rc)


def moe_check_dims(d: MoeDims) -> int:
    return load().moe_check_dims(ctypes.byref(d))


def moe_workspace_bytes(d: MoeDims) -> int:
    n = load().moe_workspace_bytes(ctypes.byref(d))
    if n == 0:
        raise MoeError("moe_workspace_bytes", moe_check_dims(d))
    return n


def alloc_workspace(d: MoeDims, device=None) -> torch.Tensor:
    """A zero-filled uint8 workspace of moe_workspace_bytes(d) bytes."""
    return torch.zeros(moe_workspace_bytes(d), dtype=torch.uint8, device=device or "cuda")


def moe_ws_init(ws: torch.Tensor, stream=None) -> None:
    _call("moe_ws_init", _ptr(ws), ws.numel(), _stream(stream))


def moe_ws_read_error(ws: torch.Tensor, clear: bool = False, stream=None) -> int:
    bits = ctypes.c_uint32(0)
    _call("moe_ws_read_error", _ptr(ws), ws.numel(), 1 if clear else 0, _stream(stream), ctypes.byref(bits))
    return bits.value


def moe_route(d: MoeDims, hidden, router_w, expert_bias, topk_idx, topk_w, ws=None, logits_out=None,
              stream=None) -> None:
    _check(hidden, torch.bfloat16, (d.T, d.H), "hidden")
    _check(router_w, torch.float32, (d.E, d.H), "router_w")
    _check(expert_bias, torch.float32, (d.E,), "expert_bias")
    _check(topk_idx, torch.int32, (d.T, d.top_k), "topk_idx")
    _check(topk_w, torch.float32, (d.T, d.top_k), "topk_w")
    _check(logits_out, torch.float32, (d.T, d.E), "logits_out")
    _call("moe_route", ctypes.byref(d), _ptr(hidden), _ptr(router_w), _ptr(expert_bias), _ptr(logits_out),
          _ptr(topk_idx), _ptr(topk_w), _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream))


def moe_permute(d: MoeDims, topk_idx, counts, offsets, perm, inv_perm, ws, stream=None) -> None:
    S = d.T * d.top_k
    _check(topk_idx, torch.int32, (d.T, d.top_k), "topk_idx")
    _check(counts, torch.int32, (d.E,), "counts")
    _check(offsets, torch.int32, (d.E + 1,), "offsets")
    _check(perm, torch.int32, (S,), "perm")
    _check(inv_perm, torch.int32, (S,), "inv_perm")
    _call("moe_permute", ctypes.byref(d), _ptr(topk_idx), _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv_perm),
          _ptr(ws), ws.numel(), _stream(stream))


def moe_expert_ffn(d: MoeDims, hidden, perm, offsets, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, y_sorted,
                   y_shared, ws, stream=None) -> None:
    S, Is = d.T * d.top_k, d.I_shared
    _check(hidden, torch.bfloat16, (d.T, d.H), "hidden")
    _check(perm, torch.int32, (S,), "perm")
    _check(offsets, torch.int32, (d.E + 1,), "offsets")
    _check(w_gate, torch.bfloat16, (d.E, d.I, d.H), "w_gate")
    _check(w_up, torch.bfloat16, (d.E, d.I, d.H), "w_up")
    _check(w_down, torch.bfloat16, (d.E, d.H, d.I), "w_down")
    _check(y_sorted, torch.bfloat16, (S, d.H), "y_sorted")
    if d.has_shared:
        _check(ws_gate, torch.bfloat16, (Is, d.H), "ws_gate")
        _check(ws_up, torch.bfloat16, (Is, d.H), "ws_up")
        _check(ws_down, torch.bfloat16, (d.H, Is), "ws_down")
        _check(y_shared, torch.bfloat16, (d.T, d.H), "y_shared")
    _call("moe_expert_ffn", ctypes.byref(d), _ptr(hidden), _ptr(perm), _ptr(offsets), _ptr(w_gate), _ptr(w_up),
          _ptr(w_down), _ptr(ws_gate), _ptr(ws_up), _ptr(ws_down), _ptr(y_sorted), _ptr(y_shared), _ptr(ws),
          ws.numel(), _stream(stream))


def moe_expert_gate_up(d: MoeDims, hidden, perm, offsets, w_gate, w_up, ws_gate, ws_up, ws, stream=None) -> None:
    _call("moe_expert_gate_up", ctypes.byref(d), _ptr(hidden), _ptr(perm), _ptr(offsets), _ptr(w_gate), _ptr(w_up),
          _ptr(ws_gate), _ptr(ws_up), _ptr(ws), ws.numel(), _stream(stream))


def moe_expert_down(d: MoeDims, offsets, w_down, ws_down, y_sorted, y_shared, ws, stream=None) -> None:
    _call("moe_expert_down", ctypes.byref(d), _ptr(offsets), _ptr(w_down), _ptr(ws_down), _ptr(y_sorted),
          _ptr(y_shared), _ptr(ws), ws.numel(), _stream(stream))


def moe_combine(d: MoeDims, y_sorted, y_shared, inv_perm, topk_w, out, stream=None) -> None:
    S = d.T * d.top_k
    _check(y_sorted, torch.bfloat16, (S, d.H), "y_sorted")
    if d.has_shared:
        _check(y_shared, torch.bfloat16, (d.T, d.H), "y_shared")
    _check(inv_perm, torch.int32, (S,), "inv_perm")
    _check(topk_w, torch.float32, (d.T, d.top_k), "topk_w")
    _check(out, torch.bfloat16, (d.T, d.H), "out")
    _call("moe_combine", ctypes.byref(d), _ptr(y_sorted), _ptr(y_shared), _ptr(inv_perm), _ptr(topk_w), _ptr(out),
          _stream(stream))


def moe_layer_forward(d: MoeDims, hidden, router_w, expert_bias, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, out,
                      ws, stream=None) -> None:
    _check(hidden, torch.bfloat16, (d.T, d.H), "hidden")
    _check(router_w, torch.float32, (d.E, d.H), "router_w")
    _check(expert_bias, torch.float32, (d.E,), "expert_bias")
    _check(w_gate, torch.bfloat16, (d.E, d.I, d.H), "w_gate")
    _check(w_up, torch.bfloat16, (d.E, d.I, d.H), "w_up")
    _check(w_down, torch.bfloat16, (d.E, d.H, d.I), "w_down")
    _check(out, torch.bfloat16, (d.T, d.H), "out")
    if d.has_shared:
        _check(ws_gate, torch.bfloat16, (d.I_shared, d.H), "ws_gate")
        _check(ws_up, torch.bfloat16, (d.I_shared, d.H), "ws_up")
        _check(ws_down, torch.bfloat16, (d.H, d.I_shared), "ws_down")
    _call("moe_layer_forward", ctypes.byref(d), _ptr(hidden), _ptr(router_w), _ptr(expert_bias), _ptr(w_gate),
          _ptr(w_up), _ptr(w_down), _ptr(ws_gate), _ptr(ws_up), _ptr(ws_down), _ptr(out), _ptr(ws), ws.numel(),
          _stream(stream))


def moe_fused_moe(d: MoeDims, hidden, topk_idx, topk_w, w_gate_up, w_down, ws_gate_up, ws_down, out, ws,
                  stream=None) -> None:
    _check(hidden, torch.bfloat16, (d.T, d.H), "hidden")
    _check(topk_idx, torch.int32, (d.T, d.top_k), "topk_idx")
    _check(topk_w, torch.float32, (d.T, d.top_k), "topk_w")
    _check(w_gate_up, torch.bfloat16, (d.E, 2 * d.I, d.H), "w_gate_up")
    _check(w_down, torch.bfloat16, (d.E, d.H, d.I), "w_down")
    _check(out, torch.bfloat16, (d.T, d.H), "out")
    if d.has_shared:
        _check(ws_gate_up, torch.bfloat16, (2 * d.I_shared, d.H), "ws_gate_up")
        _check(ws_down, torch.bfloat16, (d.H, d.I_shared), "ws_down")
    _call("moe_fused_moe", ctypes.byref(d), _ptr(hidden), _ptr(topk_idx), _ptr(topk_w), _ptr(w_gate_up), _ptr(w_down),
          _ptr(ws_gate_up), _ptr(ws_down), _ptr(out), _ptr(ws), ws.numel(), _stream(stream))


def fused_moe(hidden, topk_index, topk_weight, w_gate_up, w_down, output=None, ws_gate_up=None, ws_down=None,
              workspace=None, stream=None):
    """The fused-MoE call in the form the HunyuanImage 3.0 post shows it:
    flattened tokens [T, H] bf16, top-k indices [T, k] int32 and weights [T, k]
    fp32, stacked w_gate_up [E, 2I, H] (gate rows first) and w_down [E, H, I];
    optional shared expert ws_gate_up [2 I_s, H], ws_down [H, I_s] (added
    unweighted).  Returns `output` ([T, H] bf16, allocated when None)."""
    T, H = hidden.shape
    E, two_i, _ = w_gate_up.shape
    k = topk_index.shape[1]
    has_shared = ws_gate_up is not None
    d = dims(T, H, E, two_i // 2, k, I_shared=(ws_gate_up.shape[0] // 2) if has_shared else 0,
             score_mode="softmax", route_scale=1.0, has_shared=has_shared)
    if output is None:
        output = torch.empty((T, H), dtype=torch.bfloat16, device=hidden.device)
    if workspace is None:
        workspace = alloc_workspace(d, hidden.device)
    moe_fused_moe(d, hidden, topk_index, topk_weight, w_gate_up, w_down, ws_gate_up, ws_down, output, workspace,
                  stream)
    return output


def moe_quantize_fp8_rows(src, codes, scales, stream=None) -> None:
    """codes [R, C] uint8 (E4M3) and scales [R] fp32 of a bf16 matrix [R, C] (any
    leading dims are rows)."""
    C = src.shape[-1]
    R = src.numel() // C if C else 0
    _check(src, torch.bfloat16, src.shape, "src")
    _check(codes, torch.uint8, src.shape, "codes")
    _check(scales, torch.float32, src.shape[:-1], "scales")
    _call("moe_quantize_fp8_rows", _ptr(src), R, C, _ptr(codes), _ptr(scales), _stream(stream))


class Fp8Experts:
    """Device tensors of FP8 expert weights (E4M3 codes + one fp32 scale per
    row) and the C struct that points at them."""

    NAMES = ("gate", "up", "down", "s_gate", "s_up", "s_down")

    def __init__(self, **tensors):
        self.t = tensors  # name -> (codes uint8, scales fp32) or None
        st = MoeFp8Experts()
        for n in self.NAMES:
            pair = tensors.get(n)
            setattr(st, n, pair[0].data_ptr() if pair is not None else None)
            setattr(st, n + "_scale", pair[1].data_ptr() if pair is not None else None)
        self.struct = st


def quantize_fp8_experts(w_gate, w_up, w_down, ws_gate=None, ws_up=None, ws_down=None, stream=None) -> Fp8Experts:
    """Quantise bf16 expert weights (and the shared expert's, if given) with
    moe_quantize_fp8_rows on the device."""
    out = {}
    for n, w in (("gate", w_gate), ("up", w_up), ("down", w_down), ("s_gate", ws_gate), ("s_up", ws_up),
                 ("s_down", ws_down)):
        if w is None:
            continue
        codes = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
        scales = torch.empty(w.shape[:-1], dtype=torch.float32, device=w.device)
        moe_quantize_fp8_rows(w, codes, scales, stream)
        out[n] = (codes, scales)
    return Fp8Experts(**out)


def moe_expert_ffn_fp8(d: MoeDims, hidden, perm, offsets, w: Fp8Experts, y_sorted, y_shared, ws, stream=None) -> None:
    S = d.T * d.top_k
    _check(hidden, torch.bfloat16, (d.T, d.H), "hidden")
    _check(perm, torch.int32, (S,), "perm")
    _check(offsets, torch.int32, (d.E + 1,), "offsets")
    _check(y_sorted, torch.bfloat16, (S, d.H), "y_sorted")
    _check(w.t["gate"][0], torch.uint8, (d.E, d.I, d.H), "gate codes")
    _check(w.t["down"][0], torch.uint8, (d.E, d.H, d.I), "down codes")
    if d.has_shared:
        _check(y_shared, torch.bfloat16, (d.T, d.H), "y_shared")
        _check(w.t["s_gate"][0], torch.uint8, (d.I_shared, d.H), "shared gate codes")
    _call("moe_expert_ffn_fp8", ctypes.byref(d), _ptr(hidden), _ptr(perm), _ptr(offsets), ctypes.byref(w.struct),
          _ptr(y_sorted), _ptr(y_shared), _ptr(ws), ws.numel(), _stream(stream))


def moe_layer_forward_fp8(d: MoeDims, hidden, router_w, expert_bias, w: Fp8Experts, out, ws, stream=None) -> None:
    _check(hidden, torch.bfloat16, (d.T, d.H), "hidden")
    _check(router_w, torch.float32, (d.E, d.H), "router_w")
    _check(expert_bias, torch.float32, (d.E,), "expert_bias")
    _check(out, torch.bfloat16, (d.T, d.H), "out")
    _check(w.t["gate"][0], torch.uint8, (d.E, d.I, d.H), "gate codes")
    _call("moe_layer_forward_fp8", ctypes.byref(d), _ptr(hidden), _ptr(router_w), _ptr(expert_bias),
          ctypes.byref(w.struct), _ptr(out), _ptr(ws), ws.numel(), _stream(stream))


def moe_expert_ffn_w8a8(d: MoeDims, hidden, perm, offsets, w: Fp8Experts, y_sorted, y_shared, ws,
                        stream=None) -> None:
    """W8A8 expert FFN: FP8 weights and FP8 activations (hidden per token, the
    SiLU*up activation per routed slot) on the 8-bit tensor-core path."""
    S = d.T * d.top_k
    _check(hidden, torch.bfloat16, (d.T, d.H), "hidden")
    _check(perm, torch.int32, (S,), "perm")
    _check(offsets, torch.int32, (d.E + 1,), "offsets")
    _check(y_sorted, torch.bfloat16, (S, d.H), "y_sorted")
    _check(w.t["gate"][0], torch.uint8, (d.E, d.I, d.H), "gate codes")
    _check(w.t["down"][0], torch.uint8, (d.E, d.H, d.I), "down codes")
    if d.has_shared:
        _check(y_shared, torch.bfloat16, (d.T, d.H), "y_shared")
        _check(w.t["s_gate"][0], torch.uint8, (d.I_shared, d.H), "shared gate codes")
    _call("moe_expert_ffn_w8a8", ctypes.byref(d), _ptr(hidden), _ptr(perm), _ptr(offsets), ctypes.byref(w.struct),
          _ptr(y_sorted), _ptr(y_shared), _ptr(ws), ws.numel(), _stream(stream))


def moe_layer_forward_w8a8(d: MoeDims, hidden, router_w, expert_bias, w: Fp8Experts, out, ws, stream=None) -> None:
    _check(hidden, torch.bfloat16, (d.T, d.H), "hidden")
    _check(router_w, torch.float32, (d.E, d.H), "router_w")
    _check(expert_bias, torch.float32, (d.E,), "expert_bias")
    _check(out, torch.bfloat16, (d.T, d.H), "out")
    _check(w.t["gate"][0], torch.uint8, (d.E, d.I, d.H), "gate codes")
    _call("moe_layer_forward_w8a8", ctypes.byref(d), _ptr(hidden), _ptr(router_w), _ptr(expert_bias),
          ctypes.byref(w.struct), _ptr(out), _ptr(ws), ws.numel(), _stream(stream))


def moe_selftest_wait_timeout(ws: torch.Tensor, limit_ns: int, stream=None) -> None:
    _call("moe_selftest_wait_timeout", _ptr(ws), ws.numel(), limit_ns, _stream(stream))


def moe_selftest_silu(g, u, out, stream=None) -> None:
    """out = the expert epilogue's SiLU(g) * u, element-wise (fp32 device tensors)."""
    n = g.numel()
    _check(g, torch.float32, (n,), "g")
    _check(u, torch.float32, (n,), "u")
    _check(out, torch.float32, (n,), "out")
    _call("moe_selftest_silu", _ptr(g), _ptr(u), _ptr(out), n, _stream(stream))


class MoELayer:
    """One MoE FFN layer with device-resident weights and its own workspace:
    ``layer(hidden)`` runs moe_layer_forward on the current stream."""

    def __init__(self, d: MoeDims, router_w, expert_bias, w_gate, w_up, w_down, ws_gate=None, ws_up=None,
                 ws_down=None):
        self.d = d
        self.router_w, self.expert_bias = router_w, expert_bias
        self.w_gate, self.w_up, self.w_down = w_gate, w_up, w_down
        self.ws_gate, self.ws_up, self.ws_down = ws_gate, ws_up, ws_down
        self.ws = alloc_workspace(d, router_w.device)

    def __call__(self, hidden, out=None, stream=None):
        if out is None:
            out = torch.empty((self.d.T, self.d.H), dtype=torch.bfloat16, device=hidden.device)
        moe_layer_forward(self.d, hidden, self.router_w, self.expert_bias, self.w_gate, self.w_up, self.w_down,
                          self.ws_gate, self.ws_up, self.ws_down, out, self.ws, stream)
        return out
