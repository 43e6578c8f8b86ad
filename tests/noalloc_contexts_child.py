"""Child process of tests/test_zz_no_alloc.py (run on a GPU): calls
moe_expert_ffn_noalloc in two CUDA contexts that this process creates through
the driver API, one after the other (A, then B while A is still alive, then A
again), each with its own device buffers, and checks that every call equals
moe_expert_ffn with a workspace in the same context, bit for bit.  A cached
device address of the library's scratch array from the wrong context would
break that.  Prints one JSON line; exits non-zero on a mismatch."""
import ctypes
import json
import sys
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))

import oracle  # noqa: E402
import workloads as W  # noqa: E402
from expert_ffn_layer_gb300 import MoeDims, build  # noqa: E402

P = ctypes.c_void_p


def main():
    cu = ctypes.CDLL("libcuda.so.1")
    lib = ctypes.CDLL(str(build.LIB))
    lib.moe_expert_ffn.restype = ctypes.c_int
    lib.moe_expert_ffn.argtypes = [ctypes.POINTER(MoeDims)] + [P] * 12 + [ctypes.c_size_t, P]
    lib.moe_expert_ffn_noalloc.restype = ctypes.c_int
    lib.moe_expert_ffn_noalloc.argtypes = [ctypes.POINTER(MoeDims)] + [P] * 12
    lib.moe_workspace_bytes.restype = ctypes.c_size_t
    lib.moe_workspace_bytes.argtypes = [ctypes.POINTER(MoeDims)]
    cu.cuCtxCreate_v4.argtypes = [ctypes.POINTER(P), P, ctypes.c_uint, ctypes.c_int]
    cu.cuCtxSetCurrent.argtypes = [P]
    cu.cuCtxDestroy_v2.argtypes = [P]
    cu.cuCtxGetId.argtypes = [P, ctypes.POINTER(ctypes.c_ulonglong)]
    cu.cuMemAlloc_v2.argtypes = [ctypes.POINTER(ctypes.c_uint64), ctypes.c_size_t]
    cu.cuMemFree_v2.argtypes = [ctypes.c_uint64]
    cu.cuMemcpyHtoD_v2.argtypes = [ctypes.c_uint64, P, ctypes.c_size_t]
    cu.cuMemcpyDtoH_v2.argtypes = [P, ctypes.c_uint64, ctypes.c_size_t]
    cu.cuMemsetD8_v2.argtypes = [ctypes.c_uint64, ctypes.c_ubyte, ctypes.c_size_t]

    def check(rc, what):
        if rc != 0:
            raise RuntimeError(f"{what} returned {rc}")

    check(cu.cuInit(0), "cuInit")
    dev = ctypes.c_int()
    check(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")

    w = W.WORKLOADS["tiny"]
    inp = W.layer_inputs(w)
    ref = oracle.layer_forward(inp["hidden"], inp["router_w"], inp["bias"], inp["w_gate"], inp["w_up"],
                               inp["w_down"], inp["ws_gate"], inp["ws_up"], inp["ws_down"], top_k=w.top_k,
                               score_mode=w.score_mode, route_scale=w.route_scale, renorm_eps=w.renorm_eps)
    d = MoeDims(w.T, w.H, w.E, w.I, w.I_shared, w.top_k, 0, w.route_scale, w.renorm_eps, 1)
    S = w.T * w.top_k
    host = {"hidden": inp["hidden"], "perm": ref["perm"].astype(np.int32), "offsets": ref["offsets"].astype(np.int32),
            "w_gate": inp["w_gate"], "w_up": inp["w_up"], "w_down": inp["w_down"], "ws_gate": inp["ws_gate"],
            "ws_up": inp["ws_up"], "ws_down": inp["ws_down"]}
    out_bytes = {"y": S * w.H * 2, "z": w.T * w.H * 2}

    def run_in(ctx, tag):
        check(cu.cuCtxSetCurrent(ctx), "cuCtxSetCurrent")
        ptrs = []

        def alloc(nbytes):
            p = ctypes.c_uint64()
            check(cu.cuMemAlloc_v2(ctypes.byref(p), max(nbytes, 256)), "cuMemAlloc")
            ptrs.append(p.value)
            return p.value

        dp = {}
        for k, a in host.items():
            a = np.ascontiguousarray(a)
            dp[k] = alloc(a.nbytes)
            check(cu.cuMemcpyHtoD_v2(dp[k], a.ctypes.data, a.nbytes), "cuMemcpyHtoD")
        ws_bytes = lib.moe_workspace_bytes(ctypes.byref(d))
        ws = alloc(ws_bytes)
        check(cu.cuMemsetD8_v2(ws, 0, ws_bytes), "cuMemsetD8")
        y_ref, z_ref, y, z = (alloc(out_bytes[n]) for n in ("y", "z", "y", "z"))
        args = [dp[k] for k in ("hidden", "perm", "offsets", "w_gate", "w_up", "w_down", "ws_gate", "ws_up",
                                "ws_down")]
        check(lib.moe_expert_ffn(ctypes.byref(d), *args, y_ref, z_ref, ws, ws_bytes, None), "moe_expert_ffn")

        def fetch(p, n):
            h = np.empty(n // 2, dtype=np.uint16)
            check(cu.cuCtxSynchronize(), "cuCtxSynchronize")
            check(cu.cuMemcpyDtoH_v2(h.ctypes.data, p, n), "cuMemcpyDtoH")
            return h

        want_y, want_z = fetch(y_ref, out_bytes["y"]), fetch(z_ref, out_bytes["z"])
        same = []
        for call in range(2):
            check(cu.cuMemsetD8_v2(y, 0xFF, out_bytes["y"]), "cuMemsetD8")
            check(cu.cuMemsetD8_v2(z, 0xFF, out_bytes["z"]), "cuMemsetD8")
            check(lib.moe_expert_ffn_noalloc(ctypes.byref(d), *args, y, z, None), "moe_expert_ffn_noalloc")
            got_y, got_z = fetch(y, out_bytes["y"]), fetch(z, out_bytes["z"])
            same.append(bool(np.array_equal(got_y, want_y) and np.array_equal(got_z, want_z)))
        for p in ptrs:
            check(cu.cuMemFree_v2(p), "cuMemFree")
        return {"tag": tag, "calls_equal": same}

    ctx_a, ctx_b = P(), P()
    check(cu.cuCtxCreate_v4(ctypes.byref(ctx_a), None, 0, dev), "cuCtxCreate A")
    results = [run_in(ctx_a, "A")]
    check(cu.cuCtxCreate_v4(ctypes.byref(ctx_b), None, 0, dev), "cuCtxCreate B")
    results.append(run_in(ctx_b, "B"))
    results.append(run_in(ctx_a, "A again"))
    ids = []
    for c in (ctx_a, ctx_b):
        i = ctypes.c_ulonglong()
        check(cu.cuCtxGetId(c, ctypes.byref(i)), "cuCtxGetId")
        ids.append(i.value)
    check(cu.cuCtxSetCurrent(None), "cuCtxSetCurrent")
    check(cu.cuCtxDestroy_v2(ctx_b), "cuCtxDestroy B")
    check(cu.cuCtxDestroy_v2(ctx_a), "cuCtxDestroy A")
    ok = ids[0] != ids[1] and all(all(r["calls_equal"]) for r in results)
    print(json.dumps({"ok": ok, "context_ids": ids, "runs": results}))
    sys.exit(0 if ok else 1)


if __name__ == "__main__":
    main()
