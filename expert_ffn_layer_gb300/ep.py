"""Expert-parallel (EP) plan of the MoE layer across G GPUs: host-side logic.

The routed experts are split across G ranks by ownership (rank r holds the
contiguous experts [b[r], b[r+1]) and only their weights); every rank keeps a
replica of the router and of the shared expert, and attention-side data
parallelism gives each rank its own tokens.  Two exchange schemes move token
rows to the experts' owners and expert outputs back:

* AG-RS (AllGather + ReduceScatter): every rank gathers all ranks' hidden rows
  and routing [T, H], runs its own experts on the slots routed to them, forms a
  partial combined output for all T tokens, and a ReduceScatter sums the
  partials and hands each rank its own tokens' rows.  About 2 T H elements
  cross each rank's links per layer, whatever top_k is.
* Double all-to-all: every rank sends each of its routed slots' hidden rows to
  the owner of the slot's expert, owners run the grouped experts on what they
  receive, and a second all-to-all returns the expert outputs to the slots'
  ranks, which combine them locally.  About 2 T_local k H elements per rank.

The Ascend deployment article ("Hy3 on CANN NPUs", section 8.1, the MoE EP
table) compares the two by communicated volume and prefers AG-RS when top_k
exceeds ep_size (its case: top_k = 8, ep_size = 4), the all-to-all pair for
large EP; the Hy3 Preview case (section 9) uses MoE EP with attention DP for
decode.  The comparison operators of that table are lost in the page text; the
reading here is the plain one its own example supports: AG-RS when
top_k > ep_size.  The shared expert is replicated and applied to each rank's
own tokens after the exchange, so it never crosses a link (the article runs it
on a side stream; here it is a segment of the local expert kernel).

This module plans (ownership, slot lists, send/receive orders, buffer sizes,
bytes per exchange).  Nothing here moves data or computes the layer.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def expert_bounds(E: int, G: int) -> np.ndarray:
    """Ownership boundaries [G + 1]: rank r owns experts [b[r], b[r + 1]); the
    first E % G ranks hold one expert more."""
    if G <= 0 or E < G:
        raise ValueError(f"cannot split {E} experts over {G} ranks")
    sizes = np.full(G, E // G, dtype=np.int64)
    sizes[: E % G] += 1
    return np.concatenate([[0], np.cumsum(sizes)])


def expert_owner(E: int, G: int) -> np.ndarray:
    """owner[e] = the rank holding expert e."""
    b = expert_bounds(E, G)
    return np.searchsorted(b, np.arange(E), side="right") - 1


def choose_scheme(top_k: int, ep_size: int) -> str:
    """'none' for one rank; AG-RS when top_k > ep_size, else the all-to-all pair."""
    if ep_size <= 1:
        return "none"
    return "ag_rs" if top_k > ep_size else "all_to_all"


def exchange_elements(scheme: str, tokens_per_rank: int, H: int, top_k: int, G: int) -> int:
    """Elements one rank sends per layer in the exchange (receives are the same
    on average): AG-RS sends its T_local rows to G-1 ranks and its partial rows
    of the other ranks' tokens; the all-to-all pair sends its slots routed to
    other ranks' experts and returns the outputs of the slots it received,
    about T_local k (G-1) / G rows each way under even routing."""
    if scheme == "none":
        return 0
    T = tokens_per_rank * G
    if scheme == "ag_rs":
        return (tokens_per_rank * (G - 1) + (T - tokens_per_rank)) * H
    if scheme == "all_to_all":
        return 2 * tokens_per_rank * top_k * (G - 1) // G * H
    raise ValueError(scheme)


@dataclass
class LocalExperts:
    """The slots one rank computes, grouped by its local experts.

    slots    flat slot ids (t * k + j of the gathered batch) routed to this rank's
             experts, grouped by expert, ascending slot order within an expert
    counts   [n_local] slots per local expert; offsets [n_local + 1]
    first    the rank's first global expert id (local expert i is first + i)"""

    slots: np.ndarray
    counts: np.ndarray
    offsets: np.ndarray
    first: int


def local_slots(topk_idx: np.ndarray, E: int, G: int, rank: int) -> LocalExperts:
    """AG-RS: of the gathered routing [T, k], the slots this rank's experts serve,
    in the order the local permutation would place them (one contiguous range
    per local expert, stable by slot)."""
    b = expert_bounds(E, G)
    lo, hi = int(b[rank]), int(b[rank + 1])
    flat = np.asarray(topk_idx, dtype=np.int64).reshape(-1)
    mine = np.nonzero((flat >= lo) & (flat < hi))[0]
    order = np.argsort(flat[mine], kind="stable")
    slots = mine[order]
    counts = np.bincount(flat[slots] - lo, minlength=hi - lo).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    return LocalExperts(slots=slots, counts=counts, offsets=offsets, first=lo)


@dataclass
class DispatchPlan:
    """All-to-all dispatch of one rank's routed slots.

    send_slots   this rank's flat slots (t * k + j of its own batch) in send
                 order: grouped by destination rank, then by expert, ascending
                 slot order within an expert
    send_counts  [G] rows sent to each rank (send_slots split in that order)
    send_expert  the global expert of each sent row"""

    send_slots: np.ndarray
    send_counts: np.ndarray
    send_expert: np.ndarray


def dispatch_plan(topk_idx: np.ndarray, E: int, G: int) -> DispatchPlan:
    """Send order of a rank's own routing [T_local, k]: by (owner, expert, slot)."""
    flat = np.asarray(topk_idx, dtype=np.int64).reshape(-1)
    owner = expert_owner(E, G)
    order = np.lexsort((np.arange(flat.size), flat, owner[flat]))  # last key sorts first
    return DispatchPlan(send_slots=order, send_counts=np.bincount(owner[flat], minlength=G).astype(np.int64),
                        send_expert=flat[order])


def receive_grouping(recv_expert: np.ndarray, E: int, G: int, rank: int) -> LocalExperts:
    """The receiving side of the dispatch: rows arrive grouped by source rank (each
    source's rows sorted by expert); this groups them by local expert, stable in
    arrival order, as positions into the receive buffer."""
    b = expert_bounds(E, G)
    lo, hi = int(b[rank]), int(b[rank + 1])
    e = np.asarray(recv_expert, dtype=np.int64)
    if e.size and (e.min() < lo or e.max() >= hi):
        raise ValueError("a received row's expert is not owned by this rank")
    order = np.argsort(e - lo, kind="stable")
    counts = np.bincount(e - lo, minlength=hi - lo).astype(np.int64)
    return LocalExperts(slots=order, counts=counts, offsets=np.concatenate([[0], np.cumsum(counts)]), first=lo)


def buffer_rows(scheme: str, tokens_per_rank: int, top_k: int, G: int) -> dict:
    """Rows of H values each buffer needs per rank (worst case for the
    all-to-all receive: every slot of every rank routed to this rank's experts,
    bounded by its experts serving each token at most min(k, experts held) times)."""
    T = tokens_per_rank * G
    if scheme == "ag_rs":
        return {"gathered_hidden": T, "partial_out": T, "expert_rows": T * top_k}
    if scheme == "all_to_all":
        return {"send": tokens_per_rank * top_k, "receive_worst": T * top_k, "returned": tokens_per_rank * top_k}
    return {}
