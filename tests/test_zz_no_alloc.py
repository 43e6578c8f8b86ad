"""moe_expert_ffn_noalloc: the expert-FFN entry point for callers that cannot
allocate device memory (it keeps its scratch in the library's own device
array).  Its results must equal those of moe_expert_ffn, which takes a
caller-allocated workspace, on every call: the array is shared between calls
and keeps the previous call's contents."""
import ctypes
import json
import subprocess
import sys
from pathlib import Path

import numpy as np
import pytest
import torch

import expert_ffn_layer_gb300 as moe
import oracle
import workloads as W
from moe_testlib import LAYER_MAX_ABS, LAYER_REL_L2, DeviceLayer, dims_of, host_f64, i32_dev, rel_l2

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    import __graft_entry__

    __graft_entry__.build()
    lib = moe.load()
    f = lib.moe_expert_ffn_noalloc
    P = ctypes.c_void_p
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(moe.MoeDims)] + [P] * 12
    return f


def _ptr(t):
    return None if t is None else t.data_ptr()


# A batch whose whole-layer workspace (with y_sorted [T * top_k, H]) is beyond
# 32 MiB while the entry point's own scratch (header + activations) fits.
BEYOND_LAYER_WS = W.Workload("noalloc_wide", 600, 4096, 16, 8, 256, 256, "sigmoid", 2.826, 0.0, True, "normal", 0.1,
                             12)


@pytest.mark.parametrize("name", ["tiny", "decode", "noalloc_wide"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    f = _noalloc_fn()
    w = BEYOND_LAYER_WS if name == "noalloc_wide" else W.WORKLOADS[name]
    if name == "noalloc_wide":
        assert moe.moe_workspace_bytes(dims_of(w)) > 32 << 20
    inp = W.layer_inputs(w)
    ref = oracle.layer_forward(inp["hidden"], inp["router_w"], inp["bias"], inp["w_gate"], inp["w_up"],
                               inp["w_down"], inp["ws_gate"], inp["ws_up"], inp["ws_down"], top_k=w.top_k,
                               score_mode=w.score_mode, route_scale=w.route_scale, renorm_eps=w.renorm_eps)
    dl = DeviceLayer(w, inp)
    perm, offsets = i32_dev(ref["perm"]), i32_dev(ref["offsets"])
    y_ref, z_ref = dl.expert_ffn(perm, offsets)  # the workspace entry point
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        y = torch.full_like(y_ref, float("nan"))
        z = torch.full_like(z_ref, float("nan"))
        rc = f(ctypes.byref(dl.d), _ptr(dl.hidden), _ptr(perm), _ptr(offsets), _ptr(dl.w_gate), _ptr(dl.w_up),
               _ptr(dl.w_down), _ptr(dl.ws_gate), _ptr(dl.ws_up), _ptr(dl.ws_down), _ptr(y), _ptr(z), stream)
        assert rc == 0, moe.status_string(rc)
        torch.cuda.synchronize()
        for got, want, what in ((y, y_ref, "y_sorted"), (z, z_ref, "y_shared")):
            g, r = host_f64(got), host_f64(want)
            assert np.isfinite(g).all(), f"call {call}: {what} not finite"
            assert rel_l2(g, r) <= LAYER_REL_L2 and np.abs(g - r).max() <= LAYER_MAX_ABS, (call, what)
            # same kernels, same inputs: the results are in fact identical
            assert torch.equal(got.view(torch.int16), want.view(torch.int16)), (call, what)


def test_noalloc_rejects_dims_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    f = _noalloc_fn()
    d = dims_of(W.WORKLOADS["prefill"])  # its activations alone are ~113 MB, beyond the built-in 32 MiB
    p = ctypes.c_void_p(1 << 20)       # aligned and never dereferenced: the call fails before any launch
    rc = f(ctypes.byref(d), *([p] * 10), p, None)
    assert rc == 3, moe.status_string(rc)  # MOE_ERR_WORKSPACE


def test_noalloc_in_two_contexts_of_one_device():
    """The scratch array's device address belongs to a CUDA context, not to a
    device ordinal: a process that makes two contexts of its own current in
    turn gets correct results in each (a child process, so that the contexts it
    creates and destroys are its own)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _noalloc_fn()  # built
    child = Path(__file__).with_name("noalloc_contexts_child.py")
    r = subprocess.run([sys.executable, str(child)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["ok"] and len(set(res["context_ids"])) == 2, res
