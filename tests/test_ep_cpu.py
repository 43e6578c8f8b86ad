"""Expert-parallel plan (expert_ffn_layer_gb300.ep) on two gloo ranks: each rank
owns half of the routed experts and its own half of the tokens; the exchange
of both schemes (AllGather + ReduceScatter, and the all-to-all pair) runs for
real over torch.distributed, with each rank's experts computed by the oracle.
The sum of the ranks' work must reproduce the full oracle layer.  Unmeasured
on hardware: every box here has one GPU."""
import json
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from expert_ffn_layer_gb300 import ep


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import oracle
    import workloads as W

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = W.WORKLOADS["tiny"]  # T = 16, H = 256, E = 16, k = 4, I = 128, shared expert
    inp = W.layer_inputs(w)
    full = oracle.layer_forward(inp["hidden"], inp["router_w"], inp["bias"], inp["w_gate"], inp["w_up"],
                                inp["w_down"], inp["ws_gate"], inp["ws_up"], inp["ws_down"], top_k=w.top_k)
    Tl = w.T // world
    mine = np.arange(rank * Tl, (rank + 1) * Tl)
    x_all = W.bf16_to_f64(inp["hidden"])
    x = x_all[mine]
    # each rank routes its own tokens (the router is replicated)
    own = oracle.layer_forward(inp["hidden"][mine], inp["router_w"], inp["bias"], inp["w_gate"], inp["w_up"],
                               inp["w_down"], inp["ws_gate"], inp["ws_up"], inp["ws_down"], top_k=w.top_k)
    idx, wts = own["idx"].astype(np.int64), own["w"]
    shared = oracle.shared_expert(inp["hidden"][mine], inp["ws_gate"], inp["ws_up"], inp["ws_down"])
    b = ep.expert_bounds(w.E, world)

    def expert_rows(rows, experts, counts):
        """The oracle's expert FFN on rows grouped by local expert."""
        y = np.zeros((rows.shape[0], w.H))
        off = 0
        for i, c in enumerate(counts):
            if c:
                e = b[rank] + i
                y[off:off + c] = oracle.swiglu(_as_bf16_bits(rows[off:off + c]), inp["w_gate"][e], inp["w_up"][e],
                                               inp["w_down"][e])
            off += c
        return y

    res = {"rank": rank}
    # ---------------- AG-RS: gather everyone's rows and routing, partial outputs, reduce-scatter
    gx = torch.empty((w.T, w.H), dtype=torch.float64)
    dist.all_gather_into_tensor(gx, torch.from_numpy(x))
    gi = torch.empty((w.T, w.top_k), dtype=torch.int64)
    dist.all_gather_into_tensor(gi, torch.from_numpy(idx))
    gw = torch.empty((w.T, w.top_k), dtype=torch.float64)
    dist.all_gather_into_tensor(gw, torch.from_numpy(wts))
    gx, gi, gw = gx.numpy(), gi.numpy(), gw.numpy()
    loc = ep.local_slots(gi, w.E, world, rank)
    y = expert_rows(gx[loc.slots // w.top_k], None, loc.counts)
    partial = np.zeros((w.T, w.H))
    np.add.at(partial, loc.slots // w.top_k, gw.reshape(-1)[loc.slots][:, None] * y)
    out_rs = torch.empty((Tl, w.H), dtype=torch.float64)
    dist.reduce_scatter_tensor(out_rs, torch.from_numpy(partial))
    out_ag = out_rs.numpy() + shared
    res["ag_rs_err"] = float(np.abs(out_ag - full["out"][mine]).max())
    all_slots = [None] * world
    dist.all_gather_object(all_slots, loc.slots.tolist())
    flat = sorted(s for part in all_slots for s in part)
    res["ag_rs_slots_partition"] = flat == list(range(w.T * w.top_k))

    # ---------------- all-to-all pair: dispatch slots to owners, return outputs
    plan = ep.dispatch_plan(idx, w.E, world)
    recv_counts = torch.empty(world, dtype=torch.int64)
    dist.all_to_all_single(recv_counts, torch.from_numpy(plan.send_counts))
    rc = recv_counts.tolist()
    sc = plan.send_counts.tolist()
    send_rows = torch.from_numpy(np.ascontiguousarray(x[plan.send_slots // w.top_k]))
    recv_rows = torch.empty((sum(rc), w.H), dtype=torch.float64)
    dist.all_to_all_single(recv_rows, send_rows, output_split_sizes=rc, input_split_sizes=sc)
    recv_expert = torch.empty(sum(rc), dtype=torch.int64)
    dist.all_to_all_single(recv_expert, torch.from_numpy(plan.send_expert), output_split_sizes=rc,
                           input_split_sizes=sc)
    grp = ep.receive_grouping(recv_expert.numpy(), w.E, world, rank)
    y_grouped = expert_rows(recv_rows.numpy()[grp.slots], None, grp.counts)
    y_recv = np.empty_like(y_grouped)
    y_recv[grp.slots] = y_grouped  # back to arrival order
    back = torch.empty((int(sum(sc)), w.H), dtype=torch.float64)
    dist.all_to_all_single(back, torch.from_numpy(y_recv), output_split_sizes=sc, input_split_sizes=rc)
    y_slot = np.empty((Tl * w.top_k, w.H))
    y_slot[plan.send_slots] = back.numpy()
    out_a2a = (y_slot.reshape(Tl, w.top_k, w.H) * wts[:, :, None]).sum(axis=1) + shared
    res["a2a_err"] = float(np.abs(out_a2a - full["out"][mine]).max())
    res["a2a_sent"] = int(sum(sc))
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)
    dist.destroy_process_group()


def _as_bf16_bits(rows):
    """The gathered rows are bf16 values held in float64: back to bf16 bits (exact)."""
    return (rows.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_two_gloo_ranks_reproduce_the_layer_with_both_schemes(tmp_path):
    mp.spawn(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        res = json.loads((tmp_path / f"rank{r}.json").read_text())
        assert res["ag_rs_slots_partition"]
        assert res["ag_rs_err"] < 1e-12, res
        assert res["a2a_err"] < 1e-12, res
        assert res["a2a_sent"] == 8 * 4  # every local slot is sent once (to its expert's owner, possibly itself)


def test_ownership_and_scheme_choice():
    assert ep.expert_bounds(192, 16).tolist() == list(range(0, 193, 12))  # 12 experts per rank
    b = ep.expert_bounds(10, 4)
    assert b.tolist() == [0, 3, 6, 8, 10]
    assert ep.expert_owner(10, 4).tolist() == [0, 0, 0, 1, 1, 1, 2, 2, 3, 3]
    with pytest.raises(ValueError):
        ep.expert_bounds(3, 4)
    # the article's case: top_k = 8 over 4 ranks gathers; large EP goes all-to-all
    assert ep.choose_scheme(8, 4) == "ag_rs"
    assert ep.choose_scheme(8, 16) == "all_to_all"
    assert ep.choose_scheme(8, 1) == "none"


def test_exchange_volumes_favour_the_chosen_scheme():
    """Under even routing the chosen scheme moves no more data than the other."""
    for G in (2, 4, 8, 16, 32):
        for k in (2, 4, 8):
            ag = ep.exchange_elements("ag_rs", 1024, 4096, k, G)
            a2a = ep.exchange_elements("all_to_all", 1024, 4096, k, G)
            pick = ep.choose_scheme(k, G)
            if k > G:
                assert pick == "ag_rs" and ag <= a2a, (G, k, ag, a2a)
            elif k < G - 1:
                assert pick == "all_to_all" and a2a <= ag, (G, k, ag, a2a)


def test_dispatch_and_receive_orders():
    rng = np.random.default_rng(3)
    E, G, T, k = 12, 3, 10, 3
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    plan = ep.dispatch_plan(idx, E, G)
    flat = idx.reshape(-1)
    owner = ep.expert_owner(E, G)
    assert sorted(plan.send_slots.tolist()) == list(range(T * k))
    keys = [(owner[flat[s]], flat[s], s) for s in plan.send_slots]
    assert keys == sorted(keys)
    assert plan.send_counts.tolist() == [int((owner[flat] == r).sum()) for r in range(G)]
    recv = plan.send_expert[plan.send_counts[0]:plan.send_counts[0] + plan.send_counts[1]]
    grp = ep.receive_grouping(recv, E, G, 1)
    assert (np.diff(recv[grp.slots]) >= 0).all() and grp.counts.sum() == recv.size
    with pytest.raises(ValueError):
        ep.receive_grouping(np.array([0]), E, G, 1)
