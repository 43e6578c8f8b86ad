"""GPU parity of the FP8 (E4M3, one scale per row) expert-weight path against
the oracle: the device quantiser bit for bit, then the expert FFN and the whole
layer against the oracle's layer on the oracle's own dequantised weights
(value(code) * scale, exactly)."""
import numpy as np
import pytest
import torch

import expert_ffn_layer_gb300 as moe
import oracle
import workloads as W
from moe_testlib import DeviceLayer, assert_layer_close, bf16_dev, host_f64, i32_dev
from test_gpu_parity import MID, MID_SOFTMAX, NOSHARED, ODD_H, WIDE, _check_layer_rows, inputs_of

pytestmark = pytest.mark.gpu

WEIGHTS = ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


class _LazyExperts:
    """Stacked expert weights [E, rows, cols] whose expert e is quantised and
    dequantised by the oracle when first indexed: the oracle's expert loop only
    touches the experts a routing selects (a Hy3 layer holds 3.6 G weights)."""

    def __init__(self, src):
        self.src, self.cache = src, {}
        self.shape = src.shape

    def __getitem__(self, e):
        e = int(e)
        if e not in self.cache:
            self.cache[e] = oracle.dequantize_rows_e4m3(*oracle.quantize_rows_e4m3(self.src[e]))
        return self.cache[e]


_deq_cache = {}


def _dequantised(w, inp):
    """The inputs with every expert weight replaced by the oracle's dequantised
    FP8 weight (float64 holding bf16 values); routed experts lazily."""
    if w.name not in _deq_cache:
        out = dict(inp)
        for k in ("w_gate", "w_up", "w_down"):
            out[k] = _LazyExperts(inp[k])
        for k in ("ws_gate", "ws_up", "ws_down"):
            if inp.get(k) is not None:
                out[k] = oracle.dequantize_rows_e4m3(*oracle.quantize_rows_e4m3(inp[k]))
        _deq_cache[w.name] = out
    return _deq_cache[w.name]


def _fp8_dev(dl):
    return moe.quantize_fp8_experts(dl.w_gate, dl.w_up, dl.w_down, dl.ws_gate, dl.ws_up, dl.ws_down)


def test_quantize_rows_bit_exact():
    """Codes and scales equal the oracle's: ordinary rows, a zero row, a row
    with negative zeros, rows of tiny and of large magnitude, and exact ties."""
    w = W.normal_bf16(2, 40, (37, 512), 0.02)
    w[3] = 0
    w[4, ::2] = 0x8000                                            # -0.0
    w[5] = W.normal_bf16(2, 41, (512,), 1e-6)
    w[6] = W.normal_bf16(2, 42, (512,), 300.0)
    # a row whose values land on midpoints between E4M3 values once scaled
    pos = oracle.e4m3_value(np.arange(0x7F))
    mids = ((pos[1:-1] + pos[2:]) / 2)[:64]
    row = np.concatenate([[448.0], mids, -mids])[:128].astype(np.float32)
    w[7, :128] = (row.view(np.uint32) >> 16).astype(np.uint16)   # exact in bf16 (few significant bits)
    src = bf16_dev(w)
    codes = torch.empty(src.shape, dtype=torch.uint8, device="cuda")
    scales = torch.empty(src.shape[0], dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8_rows(src, codes, scales)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quantize_rows_e4m3(w)
    assert np.array_equal(scales.cpu().numpy(), s_ref)
    assert np.array_equal(codes.cpu().numpy(), q_ref)


def test_quantize_rows_bit_exact_wide_range():
    """The device forms each quotient w / scale from one reciprocal per row and a
    correction step; its codes equal the oracle's (fp32 division) on 2 M values
    whose rows span twelve decades of scale and whose quotients span every E4M3
    binade, subnormals included."""
    rows, cols = 1024, 2048
    rng = np.random.default_rng(7)
    row_max = 10.0 ** rng.uniform(-7, 5, size=rows)
    mag = row_max[:, None] * 2.0 ** rng.uniform(-16, 0, size=(rows, cols))
    vals = np.where(rng.random((rows, cols)) < 0.5, -mag, mag).astype(np.float32)
    vals[:, 0] = row_max.astype(np.float32)                      # the row's largest magnitude
    w = (vals.view(np.uint32) >> 16).astype(np.uint16)          # truncation to bf16 keeps |v| <= max
    src = bf16_dev(w)
    codes = torch.empty(src.shape, dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows, dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8_rows(src, codes, scales)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quantize_rows_e4m3(w)
    assert np.array_equal(scales.cpu().numpy(), s_ref)
    got = codes.cpu().numpy()
    assert np.array_equal(got, q_ref), f"{int((got != q_ref).sum())} codes differ"


@pytest.mark.parametrize("w", [W.WORKLOADS["tiny"], MID, MID_SOFTMAX, WIDE, ODD_H, NOSHARED, W.WORKLOADS["decode"]],
                         ids=["tiny", "mid", "mid_softmax", "wide", "odd_h", "noshared", "decode"])
def test_expert_ffn_fp8_parity(w):
    """Given the oracle's routing, y_sorted and y_shared match the oracle's
    expert FFN on the dequantised weights."""
    inp = inputs_of(w)
    deq = _dequantised(w, inp)
    ref = oracle.layer_forward(deq["hidden"], deq["router_w"], deq["bias"], deq["w_gate"], deq["w_up"],
                               deq["w_down"], deq.get("ws_gate"), deq.get("ws_up"), deq.get("ws_down"),
                               top_k=w.top_k, score_mode=w.score_mode, route_scale=w.route_scale,
                               renorm_eps=w.renorm_eps)
    dl = DeviceLayer(w, inp)
    fp8 = _fp8_dev(dl)
    d = dl.d
    y = torch.empty((w.S, w.H), dtype=torch.bfloat16, device="cuda")
    z = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda") if w.has_shared else None
    moe.moe_expert_ffn_fp8(d, dl.hidden, i32_dev(ref["perm"]), i32_dev(ref["offsets"]), fp8, y, z, dl.ws)
    torch.cuda.synchronize()
    assert_layer_close(host_f64(y), ref["y_sorted"], f"{w.name} fp8 y_sorted")
    if w.has_shared:
        assert_layer_close(host_f64(z), ref["z"], f"{w.name} fp8 y_shared")
    assert moe.moe_ws_read_error(dl.ws) == 0


@pytest.mark.parametrize("T", [700, 1040])
def test_expert_ffn_fp8_skewed(T):
    """One expert holding every token (several 128-token chunks), empty experts."""
    w = MID.with_(name=f"mid_fp8_{T}", T=T)
    inp = W.layer_inputs(w)
    deq = _dequantised(w, inp)
    topk = np.zeros((w.T, 2), dtype=np.int32)
    topk[:, 0] = 3
    topk[:, 1] = np.where(np.arange(w.T) < 512, 6, 1)
    counts, offsets = oracle.histogram_offsets(topk, w.E)
    perm, inv = oracle.permutation(topk, w.E)
    y_ref = oracle.expert_outputs_sorted(inp["hidden"], perm, offsets, w.top_k, deq["w_gate"], deq["w_up"],
                                         deq["w_down"])
    z_ref = oracle.shared_expert(inp["hidden"], deq["ws_gate"], deq["ws_up"], deq["ws_down"])
    dl = DeviceLayer(w, inp)
    fp8 = _fp8_dev(dl)
    y = torch.empty((w.S, w.H), dtype=torch.bfloat16, device="cuda")
    z = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_expert_ffn_fp8(dl.d, dl.hidden, i32_dev(perm), i32_dev(offsets), fp8, y, z, dl.ws)
    torch.cuda.synchronize()
    assert_layer_close(host_f64(y), y_ref, f"fp8 skewed T={T} y_sorted")
    assert_layer_close(host_f64(z), z_ref, f"fp8 skewed T={T} y_shared")
    assert moe.moe_ws_read_error(dl.ws) == 0


@pytest.mark.parametrize("w", [W.WORKLOADS["tiny"], MID, W.WORKLOADS["decode"]], ids=["tiny", "mid", "decode"])
def test_layer_fp8_parity(w):
    """moe_layer_forward_fp8 against the oracle's layer on the dequantised weights
    (near-tie routing rows compared for the selection the GPU made); repeated
    calls give the same bits."""
    inp = inputs_of(w)
    deq = _dequantised(w, inp)
    dl = DeviceLayer(w, inp)
    fp8 = _fp8_dev(dl)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_layer_forward_fp8(dl.d, dl.hidden, dl.router_w, dl.bias, fp8, out, dl.ws)
    idx, _, _ = dl.route()
    again = torch.empty_like(out)
    moe.moe_layer_forward_fp8(dl.d, dl.hidden, dl.router_w, dl.bias, fp8, again, dl.ws)
    torch.cuda.synchronize()
    _check_layer_rows(w, deq, host_f64(out), np.arange(w.T), idx.cpu().numpy())
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))
    assert moe.moe_ws_read_error(dl.ws) == 0

