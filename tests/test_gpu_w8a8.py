"""GPU parity of the W8A8 path (FP8 weights and FP8 activations on the 8-bit
tensor-core path) against the oracle's W8A8 layer: the hidden state quantised
per token, the stored bf16 SiLU(gate) * up activation per routed slot, the
weights per output row.  The oracle quantises the weights itself (the device
quantiser matches it bit for bit, tests/test_gpu_fp8.py)."""
import numpy as np
import pytest
import torch

import expert_ffn_layer_gb300 as moe
import oracle
import workloads as W
from moe_testlib import DeviceLayer, assert_layer_close, check_selection, host_f64, i32_dev, valid_alternatives
from test_gpu_parity import MID, MID_SOFTMAX, NOSHARED, inputs_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


class _LazyQuantised:
    """The oracle's E4M3 codes and scales of stacked expert weights [E, rows,
    cols], quantised expert by expert when first indexed (the oracle touches only
    the experts a routing selects)."""

    def __init__(self, src):
        self.src, self.cache = src, {}

    def _get(self, e):
        e = int(e)
        if e not in self.cache:
            self.cache[e] = oracle.quantize_rows_e4m3(self.src[e])
        return self.cache[e]

    @property
    def codes(self):
        return _Index(self, 0)

    @property
    def scales(self):
        return _Index(self, 1)


class _Index:
    def __init__(self, lazy, k):
        self.lazy, self.k = lazy, k

    def __getitem__(self, e):
        return self.lazy._get(e)[self.k]


_q_cache = {}


def _oracle_weights(w, inp):
    if w.name not in _q_cache:
        experts = tuple((lz.codes, lz.scales) for lz in (_LazyQuantised(inp[k]) for k in ("w_gate", "w_up", "w_down")))
        shared = (tuple(oracle.quantize_rows_e4m3(inp[k]) for k in ("ws_gate", "ws_up", "ws_down"))
                  if w.has_shared else None)
        _q_cache.clear()
        _q_cache[w.name] = (experts, shared)
    return _q_cache[w.name]


def _oracle_w8a8(w, inp, hidden=None, topk_idx=None):
    experts, shared = _oracle_weights(w, inp)
    return oracle.layer_forward_w8a8(inp["hidden"] if hidden is None else hidden, inp["router_w"], inp["bias"],
                                     experts, shared, top_k=w.top_k, score_mode=w.score_mode,
                                     route_scale=w.route_scale, renorm_eps=w.renorm_eps, topk_idx=topk_idx)


def _fp8_dev(dl):
    return moe.quantize_fp8_experts(dl.w_gate, dl.w_up, dl.w_down, dl.ws_gate, dl.ws_up, dl.ws_down)


# 240-token tiles with experts averaging at most 256 tokens and I = 768: the
# quantisation of each chunk split into three 256-column tiles (the shared
# expert's I = 640 into two whole blocks and a ragged one of 128 columns)
MID_WIDE_I = MID.with_(name="mid_wide_i", I=768, I_shared=640)
SHAPES = [W.WORKLOADS["tiny"], MID, MID_SOFTMAX, NOSHARED, MID_WIDE_I, W.WORKLOADS["decode"]]
SHAPE_IDS = ["tiny", "mid", "mid_softmax", "noshared", "mid_wide_i", "decode"]


@pytest.mark.parametrize("w", SHAPES, ids=SHAPE_IDS)
def test_expert_ffn_w8a8_parity(w):
    """Given the oracle's routing, y_sorted and y_shared match the oracle's W8A8
    expert FFN element by element."""
    inp = inputs_of(w)
    ref = _oracle_w8a8(w, inp)
    dl = DeviceLayer(w, inp)
    fp8 = _fp8_dev(dl)
    y = torch.empty((w.S, w.H), dtype=torch.bfloat16, device="cuda")
    z = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda") if w.has_shared else None
    moe.moe_expert_ffn_w8a8(dl.d, dl.hidden, i32_dev(ref["perm"]), i32_dev(ref["offsets"]), fp8, y, z, dl.ws)
    torch.cuda.synchronize()
    assert_layer_close(host_f64(y), ref["y_sorted"], f"{w.name} w8a8 y_sorted")
    if w.has_shared:
        assert_layer_close(host_f64(z), ref["z"], f"{w.name} w8a8 y_shared")
    assert moe.moe_ws_read_error(dl.ws) == 0


@pytest.mark.parametrize("T", [700, 1040])
def test_expert_ffn_w8a8_skewed(T):
    """One expert holding every token (several 240-token chunks), empty experts,
    a ragged last chunk."""
    w = MID.with_(name=f"mid_w8a8_{T}", T=T)
    inp = W.layer_inputs(w)
    topk = np.zeros((w.T, 2), dtype=np.int32)
    topk[:, 0] = 3
    topk[:, 1] = np.where(np.arange(w.T) < 512, 6, 1)
    ref = _oracle_w8a8(w, inp, topk_idx=topk)
    dl = DeviceLayer(w, inp)
    fp8 = _fp8_dev(dl)
    y = torch.empty((w.S, w.H), dtype=torch.bfloat16, device="cuda")
    z = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_ffn_w8a8(dl.d, dl.hidden, i32_dev(ref["perm"]), i32_dev(ref["offsets"]), fp8, y, z, dl.ws)
    torch.cuda.synchronize()
    assert_layer_close(host_f64(y), ref["y_sorted"], f"w8a8 skewed T={T} y_sorted")
    assert_layer_close(host_f64(z), ref["z"], f"w8a8 skewed T={T} y_shared")
    assert moe.moe_ws_read_error(dl.ws) == 0


@pytest.mark.parametrize("w", [W.WORKLOADS["tiny"], MID, MID_WIDE_I, W.WORKLOADS["decode"]],
                         ids=["tiny", "mid", "mid_wide_i", "decode"])
def test_layer_w8a8_parity(w):
    """moe_layer_forward_w8a8 against the oracle's W8A8 layer (near-tie rows for
    the selection the GPU made); repeated calls give the same bits."""
    inp = inputs_of(w)
    dl = DeviceLayer(w, inp)
    fp8 = _fp8_dev(dl)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_layer_forward_w8a8(dl.d, dl.hidden, dl.router_w, dl.bias, fp8, out, dl.ws)
    idx, _, _ = dl.route()
    again = torch.empty_like(out)
    moe.moe_layer_forward_w8a8(dl.d, dl.hidden, dl.router_w, dl.bias, fp8, again, dl.ws)
    torch.cuda.synchronize()
    gi = idx.cpu().numpy()
    ref = _oracle_w8a8(w, inp)
    same, ties = check_selection(gi, ref, w.top_k)
    expected = ref["out"].copy()
    for t in ties:
        g = sorted(gi[t].tolist())
        assert g in valid_alternatives(ref, t, w.top_k)
        expected[t] = _oracle_w8a8(w, inp, hidden=inp["hidden"][t:t + 1], topk_idx=np.array([g], np.int32))["out"][0]
    assert_layer_close(host_f64(out), expected, f"{w.name} w8a8 layer")
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))
    assert moe.moe_ws_read_error(dl.ws) == 0


def test_w8a8_is_close_to_the_bf16_layer():
    """The quantisation error of the whole W8A8 decode layer against the bf16
    layer stays at the E4M3 rounding level (informative bound)."""
    w = W.WORKLOADS["decode"]
    inp = inputs_of(w)
    dl = DeviceLayer(w, inp)
    fp8 = _fp8_dev(dl)
    out8 = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_layer_forward_w8a8(dl.d, dl.hidden, dl.router_w, dl.bias, fp8, out8, dl.ws)
    out16 = dl.forward()
    torch.cuda.synchronize()
    a, b = host_f64(out8), host_f64(out16)
    rel = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert rel < 0.08, rel
