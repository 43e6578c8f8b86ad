"""Seeded synthetic inputs for the MoE FFN layer: the shapes and value
distributions of the pages' workloads, shared by the oracle side and the CUDA
side of the tests and the benchmark.

This module holds none of the layer's arithmetic.  It turns (seed, tensor id,
element index) into numbers through a counter-based hash (``gen.c``) and knows
the five workload shapes.  bf16 tensors are returned as ``numpy.uint16`` bit
patterns; fp32 tensors as ``numpy.float32``.

Workloads (shapes from the Hy3 model facts on the hy3 README page, "Model
facts" table, and the HunyuanImage 3.0 MoE post, "Routed Experts" section):

=========  =====  ====  ===  ==  ====  ==========================================
name       T      H     E    k   I     routing
=========  =====  ====  ===  ==  ====  ==========================================
tiny       16     256   16   4   128   sigmoid + bias N(0, 0.1), x2.826
decode     8      4096  192  8   1536  sigmoid + bias N(0, 0.1), x2.826
prefill    4096   4096  192  8   1536  sigmoid + bias N(0, 0.1), x2.826
prefill_u  4096   4096  192  8   1536  sigmoid + bias N(0, 0.01), x2.826
zipf       16384  4096  192  8   1536  sigmoid + Zipf(1.1) bias, x2.826
image      8192   4096  64   8   3072  softmax, top-k, / clamp(sum, 1e-8)
=========  =====  ====  ===  ==  ====  ==========================================

Every workload has one shared expert with intermediate size I.  hidden ~ N(0,1)
bf16; expert and shared weights ~ N(0, 0.02) bf16; router weight ~ N(0, 0.02)
fp32; bias fp32.
"""
from __future__ import annotations

import ctypes
import json
import math
import os
import subprocess
import tempfile
from dataclasses import dataclass, replace
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "gen.c"
_LIB = _HERE / "_build" / "libworkloads.so"
_ZIPF_BETA = _HERE.parent / "tests" / "golden" / "zipf_beta.json"

# tensor ids: each tensor of a workload draws from its own stream
TID_HIDDEN, TID_ROUTER_W, TID_BIAS = 1, 2, 3
TID_W_GATE, TID_W_UP, TID_W_DOWN = 4, 5, 6
TID_WS_GATE, TID_WS_UP, TID_WS_DOWN = 7, 8, 9
TID_ZIPF_RANK = 10
TID_AUX = 100  # synthetic stage inputs for isolated stage tests


def build_library(force: bool = False) -> Path:
    """Compile gen.c into a shared library next to it (gcc, OpenMP, no fp contraction
    so that x86 and Arm hosts produce the same bits)."""
    if _LIB.exists() and not force and _LIB.stat().st_mtime >= _SRC.stat().st_mtime:
        return _LIB
    _LIB.parent.mkdir(exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_LIB.parent)
    os.close(fd)
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", str(_SRC), "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _get_lib():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(str(build_library()))
        u64, i64, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
        ptr = ctypes.c_void_p
        lib.wl_normal_bf16.argtypes = [u64, u64, u64, i64, dbl, dbl, ptr]
        lib.wl_normal_f32.argtypes = [u64, u64, u64, i64, dbl, dbl, ptr]
        lib.wl_uniform_f64.argtypes = [u64, u64, u64, i64, ptr]
        lib.wl_permutation.argtypes = [u64, u64, i64, ptr]
        lib.wl_randint.argtypes = [u64, u64, u64, i64, i64, ptr]
        _lib = lib
    return _lib


def normal_bf16(seed: int, tid: int, shape, sigma: float, mean: float = 0.0, offset: int = 0) -> np.ndarray:
    """N(mean, sigma^2) drawn in double and rounded once to bf16; returned as uint16 bits."""
    out = np.empty(shape, dtype=np.uint16)
    _get_lib().wl_normal_bf16(seed, tid, offset, out.size, mean, sigma, out.ctypes.data)
    return out


def normal_f32(seed: int, tid: int, shape, sigma: float, mean: float = 0.0, offset: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _get_lib().wl_normal_f32(seed, tid, offset, out.size, mean, sigma, out.ctypes.data)
    return out


def uniform_f64(seed: int, tid: int, shape, offset: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float64)
    _get_lib().wl_uniform_f64(seed, tid, offset, out.size, out.ctypes.data)
    return out


def permutation(seed: int, tid: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _get_lib().wl_permutation(seed, tid, n, out.ctypes.data)
    return out


def randint(seed: int, tid: int, shape, high: int, offset: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.int32)
    _get_lib().wl_randint(seed, tid, offset, out.size, high, out.ctypes.data)
    return out


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64 (a storage conversion)."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    top_k: int
    I: int
    I_shared: int
    score_mode: str          # "sigmoid" or "softmax"
    route_scale: float
    renorm_eps: float
    has_shared: bool
    bias: str                # "normal", "zipf" or "none"
    bias_sigma: float
    seed: int
    hidden_sigma: float = 1.0
    weight_sigma: float = 0.02
    router_sigma: float = 0.02

    @property
    def S(self) -> int:
        return self.T * self.top_k

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    def describe(self) -> dict:
        return {"workload": self.name, "T": self.T, "H": self.H, "E": self.E, "top_k": self.top_k,
                "I": self.I, "I_shared": self.I_shared if self.has_shared else 0,
                "score": self.score_mode, "bias": self.bias, "seed": self.seed}


def _hy3(name, T, seed, bias="normal", bias_sigma=0.1):
    return Workload(name, T, 4096, 192, 8, 1536, 1536, "sigmoid", 2.826, 0.0, True,
                    bias, bias_sigma, seed)


WORKLOADS = {
    "tiny": Workload("tiny", 16, 256, 16, 4, 128, 128, "sigmoid", 2.826, 0.0, True, "normal", 0.1, 0),
    "decode": _hy3("decode", 8, 1),
    "prefill": _hy3("prefill", 4096, 2),
    "prefill_u": _hy3("prefill_u", 4096, 2, bias_sigma=0.01),
    "zipf": _hy3("zipf", 16384, 3, bias="zipf"),
    "image": Workload("image", 8192, 4096, 64, 8, 3072, 3072, "softmax", 1.0, 1e-8, True, "none", 0.0, 4),
    # profiling proxies: the same tile shapes with fewer experts resident (< 2 GB of
    # weights), for hardware-counter captures that replay a kernel many times
    "decode_e48": Workload("decode_e48", 8, 4096, 48, 8, 1536, 1536, "sigmoid", 2.826, 0.0, True, "normal", 0.1, 1),
    "prefill_e32": Workload("prefill_e32", 704, 4096, 32, 8, 1536, 1536, "sigmoid", 2.826, 0.0, True, "normal", 0.1,
                            2),
}


def zipf_beta(w: Workload) -> float:
    """beta for the Zipf bias, stored by tests/golden/make_zipf_beta.py (written from the oracle's router)."""
    table = json.loads(_ZIPF_BETA.read_text())
    key = f"{w.name}:T{w.T}:E{w.E}:seed{w.seed}"
    if key not in table["beta"]:
        raise KeyError(f"no stored Zipf beta for {key}; run tests/golden/make_zipf_beta.py")
    return float(table["beta"][key])


def zipf_bias(w: Workload, beta: float) -> np.ndarray:
    """bias[e] = beta * ln(rank_e ** -1.1), rank a seeded permutation of 1..E (fp32)."""
    rank = permutation(w.seed, TID_ZIPF_RANK, w.E).astype(np.float64) + 1.0
    return (beta * (-1.1) * np.log(rank)).astype(np.float32)


def router_inputs(w: Workload, rows=None):
    """hidden (bf16 bits [T,H] or the selected rows), router_w fp32 [E,H], bias fp32 [E] or None."""
    if rows is None:
        hidden = normal_bf16(w.seed, TID_HIDDEN, (w.T, w.H), w.hidden_sigma)
    else:
        rows = np.asarray(rows, dtype=np.int64)
        hidden = np.empty((rows.size, w.H), dtype=np.uint16)
        for r, t in enumerate(rows):
            hidden[r] = normal_bf16(w.seed, TID_HIDDEN, (w.H,), w.hidden_sigma, offset=int(t) * w.H)
    router_w = normal_f32(w.seed, TID_ROUTER_W, (w.E, w.H), w.router_sigma)
    if w.bias == "normal":
        bias = normal_f32(w.seed, TID_BIAS, (w.E,), w.bias_sigma)
    elif w.bias == "zipf":
        bias = zipf_bias(w, zipf_beta(w))
    else:
        bias = None
    return hidden, router_w, bias


def expert_weights(w: Workload, experts=None):
    """Stacked routed weights: gate, up [E,I,H], down [E,H,I] (bf16 bits).

    With ``experts`` given, only those experts' slices are generated (others stay zero)."""
    E, I, H = w.E, w.I, w.H
    gate = np.zeros((E, I, H), dtype=np.uint16)
    up = np.zeros((E, I, H), dtype=np.uint16)
    down = np.zeros((E, H, I), dtype=np.uint16)
    sel = range(E) if experts is None else sorted(set(int(e) for e in experts))
    for e in sel:
        gate[e] = normal_bf16(w.seed, TID_W_GATE, (I, H), w.weight_sigma, offset=e * I * H)
        up[e] = normal_bf16(w.seed, TID_W_UP, (I, H), w.weight_sigma, offset=e * I * H)
        down[e] = normal_bf16(w.seed, TID_W_DOWN, (H, I), w.weight_sigma, offset=e * H * I)
    return gate, up, down


def shared_weights(w: Workload):
    """Shared expert: gate, up [I_s,H], down [H,I_s] (bf16 bits), or (None, None, None)."""
    if not w.has_shared:
        return None, None, None
    Is, H = w.I_shared, w.H
    return (normal_bf16(w.seed, TID_WS_GATE, (Is, H), w.weight_sigma),
            normal_bf16(w.seed, TID_WS_UP, (Is, H), w.weight_sigma),
            normal_bf16(w.seed, TID_WS_DOWN, (H, Is), w.weight_sigma))


def layer_inputs(w: Workload):
    """Everything one layer forward takes, as a dict of numpy arrays."""
    hidden, router_w, bias = router_inputs(w)
    gate, up, down = expert_weights(w)
    sg, su, sd = shared_weights(w)
    return {"hidden": hidden, "router_w": router_w, "bias": bias,
            "w_gate": gate, "w_up": up, "w_down": down,
            "ws_gate": sg, "ws_up": su, "ws_down": sd}


def synthetic_topk(w: Workload, seed_offset: int = 0) -> np.ndarray:
    """A random valid routing table [T, k] (k distinct experts per token), for
    testing the permutation and combine stages on their own."""
    T, E, k = w.T, w.E, w.top_k
    u = uniform_f64(w.seed + seed_offset, TID_AUX, (T, E))
    return np.argsort(u, axis=1, kind="stable")[:, :k].astype(np.int32)


def synthetic_weights(w: Workload, seed_offset: int = 0) -> np.ndarray:
    """Random positive combine weights [T, k] (fp32) for isolated combine tests."""
    return (uniform_f64(w.seed + seed_offset, TID_AUX + 1, (w.T, w.top_k)) + 0.05).astype(np.float32)
