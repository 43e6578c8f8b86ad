"""Helpers shared by the GPU parity tests: host<->device conversion, the C-ABI
calls on a workload, and the comparison rules."""
from __future__ import annotations

import itertools

import numpy as np
import torch

import expert_ffn_layer_gb300 as moe
import oracle
import workloads as W

# Layer tolerance (the benchmark spec): relative L2 <= 5e-3 and max |diff| <= 3e-2 against
# the fp64 oracle, bf16 storage with fp32 accumulation.
LAYER_REL_L2 = 5e-3
LAYER_MAX_ABS = 3e-2
# Router: relative error <= 1e-5 against the exact product of the same inputs.
ROUTER_REL_L2 = 1e-5
# Near-tie rule: routing may differ where the k-th and (k+1)-th keys are within 1e-5.
NEAR_TIE = 1e-5


def bf16_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def f32_dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def i32_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def dims_of(w: W.Workload, **kw):
    return moe.dims(w.T, w.H, w.E, w.I, w.top_k, w.I_shared, w.score_mode, w.route_scale, w.renorm_eps,
                    w.has_shared, **kw)


def rel_l2(got, ref) -> float:
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (n if n > 0 else 1.0))


def assert_layer_close(got, ref, what=""):
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    r = rel_l2(got, ref)
    m = float(np.abs(got - ref).max()) if got.size else 0.0
    assert r <= LAYER_REL_L2 and m <= LAYER_MAX_ABS, f"{what}: rel_l2={r:.3e} max_abs={m:.3e}"
    return r, m


class DeviceLayer:
    """A workload's inputs on the device plus a workspace."""

    def __init__(self, w: W.Workload, inp: dict):
        self.w, self.inp = w, inp
        self.d = dims_of(w)
        self.hidden = bf16_dev(inp["hidden"])
        self.router_w = f32_dev(inp["router_w"])
        self.bias = f32_dev(inp["bias"])
        self.w_gate, self.w_up, self.w_down = (bf16_dev(inp[k]) for k in ("w_gate", "w_up", "w_down"))
        if w.has_shared:
            self.ws_gate, self.ws_up, self.ws_down = (bf16_dev(inp[k]) for k in ("ws_gate", "ws_up", "ws_down"))
        else:
            self.ws_gate = self.ws_up = self.ws_down = None
        self.ws = moe.alloc_workspace(self.d)

    def route(self):
        d = self.d
        idx = torch.empty((d.T, d.top_k), dtype=torch.int32, device="cuda")
        wts = torch.empty((d.T, d.top_k), dtype=torch.float32, device="cuda")
        logits = torch.empty((d.T, d.E), dtype=torch.float32, device="cuda")
        moe.moe_route(d, self.hidden, self.router_w, self.bias, idx, wts, self.ws, logits_out=logits)
        return idx, wts, logits

    def permute(self, idx):
        d = self.d
        S = d.T * d.top_k
        counts = torch.empty(d.E, dtype=torch.int32, device="cuda")
        offsets = torch.empty(d.E + 1, dtype=torch.int32, device="cuda")
        perm = torch.empty(S, dtype=torch.int32, device="cuda")
        inv = torch.empty(S, dtype=torch.int32, device="cuda")
        moe.moe_permute(d, idx, counts, offsets, perm, inv, self.ws)
        return counts, offsets, perm, inv

    def expert_ffn(self, perm, offsets):
        d = self.d
        y = torch.empty((d.T * d.top_k, d.H), dtype=torch.bfloat16, device="cuda")
        z = torch.empty((d.T, d.H), dtype=torch.bfloat16, device="cuda") if d.has_shared else None
        moe.moe_expert_ffn(d, self.hidden, perm, offsets, self.w_gate, self.w_up, self.w_down, self.ws_gate,
                           self.ws_up, self.ws_down, y, z, self.ws)
        return y, z

    def combine(self, y, z, inv, wts):
        out = torch.empty((self.d.T, self.d.H), dtype=torch.bfloat16, device="cuda")
        moe.moe_combine(self.d, y, z, inv, wts, out)
        return out

    def forward(self):
        out = torch.empty((self.d.T, self.d.H), dtype=torch.bfloat16, device="cuda")
        moe.moe_layer_forward(self.d, self.hidden, self.router_w, self.bias, self.w_gate, self.w_up, self.w_down,
                              self.ws_gate, self.ws_up, self.ws_down, out, self.ws)
        return out


def oracle_layer(w: W.Workload, inp: dict, hidden=None, topk_idx=None):
    return oracle.layer_forward(inp["hidden"] if hidden is None else hidden, inp["router_w"], inp["bias"],
                                inp["w_gate"], inp["w_up"], inp["w_down"], inp["ws_gate"], inp["ws_up"],
                                inp["ws_down"], top_k=w.top_k, score_mode=w.score_mode, route_scale=w.route_scale,
                                renorm_eps=w.renorm_eps, topk_idx=topk_idx)


def check_selection(gpu_idx: np.ndarray, ref: dict, k: int):
    """Per row: the GPU's expert set equals the oracle's, or the row is a near tie
    and the GPU's set is one of the valid selections.  Returns (same_rows, tie_rows)."""
    mand, cand = oracle.near_tie_alternatives(ref["keys"], k, NEAR_TIE)
    same, ties = [], []
    for t in range(gpu_idx.shape[0]):
        g = set(gpu_idx[t].tolist())
        o = set(ref["idx"][t].tolist())
        assert len(g) == k, f"row {t}: duplicate experts {gpu_idx[t]}"
        if g == o:
            same.append(t)
            continue
        assert ref["margin"][t] < NEAR_TIE, f"row {t}: gpu {sorted(g)} oracle {sorted(o)} margin {ref['margin'][t]}"
        m = set(np.nonzero(mand[t])[0].tolist())
        c = set(np.nonzero(cand[t])[0].tolist())
        assert m <= g <= (m | c), f"row {t}: gpu selection {sorted(g)} is not a valid near-tie choice"
        ties.append(t)
    return same, ties


def valid_alternatives(ref: dict, t: int, k: int, limit: int = 64):
    """All valid selections of row t under the near-tie rule, from the oracle's keys."""
    mand, cand = oracle.near_tie_alternatives(ref["keys"][t:t + 1], k, NEAR_TIE)
    m = np.nonzero(mand[0])[0].tolist()
    c = np.nonzero(cand[0])[0].tolist()
    out = []
    for extra in itertools.combinations(c, k - len(m)):
        out.append(sorted(m + list(extra)))
        if len(out) >= limit:
            break
    return out
