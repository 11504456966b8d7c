"""Expert parallelism for the top-2 MoE layer: experts split over ranks, tokens moved to them.

The pages place Mixtral's experts on different devices and note that routing
decides where each token's work happens, so load follows the router: a rank
that owns popular experts is over-subscribed (fdeinterviews.com breakdown, "Why
it matters to an FDE"; lecture, router walkthrough: each token touches two of
the eight experts). This module is that layout for N ranks, each holding E/N
experts (``owner[e]`` is the rank of expert e):

1. every rank routes and groups its own tokens (``moe_route_top2``,
   ``moe_permute``): expert-contiguous rows ``x_perm`` and per-expert counts;
2. the ranks exchange their counts, so each can compute the same ``plan``;
3. dispatch: each rank sends the rows of expert e to ``owner[e]``
   (an all-to-all with per-pair row counts), the receiver regroups them by its
   own experts, source rank after source rank;
4. each rank runs its experts on what it received (``moe_expert_ffn`` with
   E/N experts and their gate weights);
5. return: the scaled expert outputs go back to the rows' source ranks (the
   reverse all-to-all), which put them back in their ``x_perm`` order and
   combine the two rows of every token (``moe_combine``).

When a rank has room for more than E/N experts' weights, ``replicated_placement``
gives the hot experts copies on several ranks (``owner[e]`` becomes a list of
ranks); each source then splits its rows of a copied expert into consecutive,
near-equal chunks, one per copy, so no single rank carries a hot expert's rows
alone. The result does not change: a row meets the same weights on any copy.

Every token gets exactly the mixture of the single-GPU layer. ``plan`` is plain
host logic. ``ExpertParallelLayer`` runs the steps over a torch.distributed
process group (NCCL on GPUs; the tests run it over gloo with CPU stand-ins for
the kernels). ``emulate`` runs N ranks' worth of the layer on one GPU with
the library's kernels, the all-to-alls becoming row gathers inside one device
buffer, to check the bookkeeping and to measure each rank's share of the
expert work under skewed routing.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def contiguous_owners(E: int, N: int) -> np.ndarray:
    """Rank r owns experts r*E/N .. (r+1)*E/N - 1."""
    if E % N:
        raise ValueError("the expert count must be a multiple of the rank count")
    return np.repeat(np.arange(N), E // N)


def balanced_owners(load, N: int) -> np.ndarray:
    """E/N experts per rank, placed to even out the rows per rank.

    Experts are taken from the most to the least loaded (ties: lower index) and
    each goes to the rank with the fewest rows so far that still has room
    (ties: lower rank) -- the longest-processing-time rule with equal capacity.
    """
    load = np.asarray(load, dtype=np.int64)
    E = load.size
    if E % N:
        raise ValueError("the expert count must be a multiple of the rank count")
    cap = E // N
    owner = np.full(E, -1, dtype=np.int64)
    rows = np.zeros(N, dtype=np.int64)
    held = np.zeros(N, dtype=np.int64)
    for e in sorted(range(E), key=lambda q: (-load[q], q)):
        free = [r for r in range(N) if held[r] < cap]
        r = min(free, key=lambda q: (rows[q], q))
        owner[e] = r
        rows[r] += load[e]
        held[r] += 1
    return owner


def _place_pieces(load, copies, N: int, slots: int):
    """Longest-processing-time placement of every expert's copies.

    Each copy of expert e carries load[e] / copies[e] rows. Copies go from the
    largest to the smallest (ties: lower expert) to the least loaded rank
    (ties: lower rank) that has a free slot and no copy of e yet. Returns the
    ranks of each expert's copies and the largest rank load, or None when the
    copies do not fit.
    """
    E = load.size
    pieces = sorted(((load[e] / copies[e], e) for e in range(E) for _ in range(copies[e])),
                    key=lambda t: (-t[0], t[1]))
    rows = np.zeros(N)
    held = np.zeros(N, dtype=np.int64)
    place = [[] for _ in range(E)]
    for size, e in pieces:
        free = [q for q in range(N) if held[q] < slots and q not in place[e]]
        if not free:
            return None
        q = min(free, key=lambda r: (rows[r], r))
        place[e].append(q)
        rows[q] += size
        held[q] += 1
    return place, rows.max()


def replicated_placement(load, N: int, slots: int) -> list:
    """Experts' copies over N ranks when a rank can hold `slots` experts' weights.

    A hot expert bounds an expert-parallel step alone once its rows exceed a
    rank's share; copies of it on several ranks split those rows. Starting from
    one copy per expert, the expert whose copies carry the most rows gets one
    more copy, while slots and ranks remain; every count of copies is placed by
    ``_place_pieces`` and the placement with the smallest largest rank load
    wins (ties: fewer copies). A replicated expert's rows are split evenly over
    its copies (``plan`` splits every source's block). Returns one list of
    ranks per expert.
    """
    load = np.asarray(load, dtype=np.float64)
    E = load.size
    if E > N * slots:
        raise ValueError("the ranks' slots cannot hold every expert once")
    copies = np.ones(E, dtype=np.int64)
    best = _place_pieces(load, copies, N, slots)
    while copies.sum() < N * slots:
        e = max(range(E), key=lambda k: (load[k] / copies[k], -k))
        if copies[e] == N or load[e] == 0:
            break
        copies[e] += 1
        got = _place_pieces(load, copies, N, slots)
        if got is not None and got[1] < best[1]:
            best = got
    return best[0]


@dataclass
class Plan:
    """Row movements of one expert-parallel step, identical on every rank.

    counts[s][e]  rows of expert e on source rank s (its x_perm rows
                  offsets[s][e] .. offsets[s][e+1])
    placement[e]  ranks holding expert e; source s's rows of e are split into
                  len(placement[e]) consecutive chunks, chunk j going to
                  placement[e][j]
    experts[q]    experts held by rank q, ascending
    send_index[s] s's x_perm rows in send order: destination by destination,
                  each destination's experts in ascending order
    send_splits[s][q], recv_splits[q][s]   rows per (source, destination)
    regroup[q]    rows of q's receive buffer in q's expert-major order (source
                  ranks in order inside each expert)
    local_offsets[q]  [len(experts[q]) + 1] group starts of q's experts
    """
    counts: np.ndarray
    offsets: np.ndarray
    placement: list
    experts: list
    send_index: list
    send_splits: np.ndarray
    recv_splits: np.ndarray
    regroup: list
    local_offsets: list

    @property
    def rows_per_rank(self) -> np.ndarray:
        return np.array([lo[-1] for lo in self.local_offsets], dtype=np.int64)

    @property
    def owner(self) -> np.ndarray:
        """The first rank of each expert (its only one without replication)."""
        return np.array([reps[0] for reps in self.placement], dtype=np.int64)


def _as_placement(owner_or_placement, E: int) -> list:
    first = owner_or_placement[0] if len(owner_or_placement) else 0
    if isinstance(first, (list, tuple)):
        return [[int(q) for q in reps] for reps in owner_or_placement]
    return [[int(q)] for q in np.asarray(owner_or_placement, dtype=np.int64)]


def plan(counts, owner) -> Plan:
    """owner: the rank of each expert, or a list of replica ranks per expert."""
    counts = np.asarray(counts, dtype=np.int64)
    N, E = counts.shape
    place = _as_placement(owner, E)
    offsets = np.zeros((N, E + 1), dtype=np.int64)
    offsets[:, 1:] = np.cumsum(counts, axis=1)
    experts = [[e for e in range(E) if q in place[e]] for q in range(N)]

    def chunk(s, e, q):
        """Rows of source s's expert-e block that go to rank q."""
        reps = place[e]
        k, j = len(reps), reps.index(q)
        c = counts[s, e]
        lo = offsets[s, e] + (c * j) // k
        hi = offsets[s, e] + (c * (j + 1)) // k
        return lo, hi

    send_index, send_splits = [], np.zeros((N, N), dtype=np.int64)
    for s in range(N):
        idx = []
        for q in range(N):
            for e in experts[q]:
                lo, hi = chunk(s, e, q)
                idx.extend(range(lo, hi))
                send_splits[s, q] += hi - lo
        send_index.append(np.array(idx, dtype=np.int64))
    recv_splits = send_splits.T.copy()
    regroup, local_offsets = [], []
    for q in range(N):
        # receive buffer of q: source after source, each source's rows in q's expert order
        start, at = {}, 0
        for s in range(N):
            for e in experts[q]:
                lo, hi = chunk(s, e, q)
                start[(s, e)] = (at, hi - lo)
                at += hi - lo
        idx, lo_off = [], [0]
        for e in experts[q]:
            for s in range(N):
                a, n = start[(s, e)]
                idx.extend(range(a, a + n))
            lo_off.append(len(idx))
        regroup.append(np.array(idx, dtype=np.int64))
        local_offsets.append(np.array(lo_off, dtype=np.int64))
    return Plan(counts, offsets, place, experts, send_index, send_splits, recv_splits, regroup, local_offsets)


def _gate_rows(perm_w):
    """Gate weights as 16-byte rows (weight, 0, 0, 0), so they move with the same row gathers."""
    import torch
    g = torch.zeros((perm_w.shape[0], 4), dtype=perm_w.dtype, device=perm_w.device)
    g[:, 0] = perm_w
    return g


def _inverse(perm: np.ndarray) -> np.ndarray:
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size, dtype=perm.dtype)
    return inv


class CudaOps:
    """The per-rank steps on this library's kernels (cuda device tensors)."""

    def __init__(self):
        from . import moe
        self.moe = moe

    def route_and_group(self, x, w_gate, E: int):
        import torch
        moe = self.moe
        T, d = x.shape
        s = moe.make_shape(T, d, 128, moe.dtype_code(x), E=E)
        i32 = dict(dtype=torch.int32, device=x.device)
        idx = torch.empty((T, 2), **i32)
        gw = torch.empty((T, 2), dtype=torch.float32, device=x.device)
        out = dict(counts=torch.empty(E, **i32), offsets=torch.empty(E + 1, **i32),
                   perm_token=torch.empty(2 * T, **i32), slot_row=torch.empty((T, 2), **i32),
                   perm_w=torch.empty(2 * T, dtype=torch.float32, device=x.device),
                   x_perm=torch.empty((2 * T, d), dtype=x.dtype, device=x.device))
        if T:
            moe.moe_route_top2(s, x, w_gate, idx, gw)
            pws = torch.empty(max(16, moe.moe_permute_workspace_bytes(s)), dtype=torch.uint8, device=x.device)
            moe.moe_permute(s, idx, gw, x, out["counts"], out["offsets"], out["perm_token"], out["slot_row"],
                            out["perm_w"], out["x_perm"], pws)
        else:
            out["counts"].zero_()
            out["offsets"].zero_()
        return out

    def gather(self, src, index):
        """Rows src[index] (index: host integers) through moe_gather_rows."""
        import torch
        index = np.asarray(index, dtype=np.int64)
        dst = torch.empty((index.size,) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device)
        if index.size:
            idx = torch.from_numpy(index.astype(np.int32)).to(src.device)
            self.moe.moe_gather_rows(src, idx, dst)
        return dst

    def experts(self, rows, local_offsets, gate, w1, w3, w2):
        """Scaled outputs gate[r] * E_e(rows[r]) of the rank's experts, fp32."""
        import torch
        moe = self.moe
        n, d = rows.shape
        E, F, _ = w1.shape
        out = torch.empty((n, d), dtype=torch.float32, device=rows.device)
        if n == 0:
            return out
        # the FFN's row buffers hold 2T rows and each expert at most T of them
        s = moe.make_shape(n, d, F, moe.dtype_code(rows), E=E)
        xp = torch.zeros((2 * n, d), dtype=rows.dtype, device=rows.device)
        xp[:n] = rows
        pw = torch.zeros(2 * n, dtype=torch.float32, device=rows.device)
        pw[:n] = gate
        ys = torch.empty((2 * n, d), dtype=torch.float32, device=rows.device)
        off = torch.as_tensor(local_offsets, dtype=torch.int32).to(rows.device)
        moe.moe_expert_ffn(s, xp, off, pw, w1, w3, w2, ys, moe.workspace(s, rows.device, ffn_only=True))
        return ys[:n]

    def combine(self, y_slot, slot_row, dtype):
        import torch
        moe = self.moe
        T = slot_row.shape[0]
        d = y_slot.shape[1]
        y = torch.empty((T, d), dtype=dtype, device=y_slot.device)
        if T:
            s = moe.make_shape(T, d, 128, moe.dtype_code(y), E=8)
            moe.moe_combine(s, y_slot, slot_row, y)
        return y


class ExpertParallelLayer:
    """One rank of an expert-parallel layer over a torch.distributed process group.

    w_gate is replicated; w1, w3, w2 hold only the experts this rank holds
    (``owner[e] == rank``, or ``rank in owner[e]`` for a replica placement),
    ascending. ``ops`` runs the per-rank steps (default: the CUDA kernels); a
    test may pass CPU stand-ins.
    """

    def __init__(self, w_gate, w1_local, w3_local, w2_local, owner, group=None, ops=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        self.E = len(owner)
        self.placement = _as_placement(owner, self.E)
        if sorted({q for reps in self.placement for q in reps}) != list(range(self.world)):
            raise ValueError("every rank must hold experts")
        self.w_gate, self.w1, self.w3, self.w2 = w_gate, w1_local, w3_local, w2_local
        self.ops = ops if ops is not None else CudaOps()
        self.last_plan = None

    def forward(self, x):
        import torch
        dist, ops = self.dist, self.ops
        g = ops.route_and_group(x, self.w_gate, self.E)
        counts = g["counts"].to(torch.int64)
        every = [torch.zeros_like(counts) for _ in range(self.world)]
        dist.all_gather(every, counts, group=self.group)
        p = plan(torch.stack(every).cpu().numpy(), self.placement)
        self.last_plan = p
        me = self.rank
        # dispatch rows and their gate weights
        send = ops.gather(g["x_perm"], p.send_index[me])
        send_w = ops.gather(_gate_rows(g["perm_w"]), p.send_index[me])
        n_in = int(p.recv_splits[me].sum())
        recv = torch.empty((n_in,) + tuple(send.shape[1:]), dtype=send.dtype, device=send.device)
        recv_w = torch.empty((n_in, 4), dtype=send_w.dtype, device=send.device)
        ins, outs = p.send_splits[me].tolist(), p.recv_splits[me].tolist()
        dist.all_to_all_single(recv, send, outs, ins, group=self.group)
        dist.all_to_all_single(recv_w, send_w, outs, ins, group=self.group)
        # this rank's experts, grouped expert by expert
        local = ops.gather(recv, p.regroup[me])
        local_w = ops.gather(recv_w, p.regroup[me])[:, 0].contiguous()
        y_local = ops.experts(local, p.local_offsets[me], local_w, self.w1, self.w3, self.w2)
        # return to the sources, back in their x_perm order, and combine
        back = ops.gather(y_local, _inverse(p.regroup[me]))
        ret = torch.empty((send.shape[0], back.shape[1]), dtype=back.dtype, device=back.device)
        dist.all_to_all_single(ret, back, ins, outs, group=self.group)
        y_slot = ops.gather(ret, _inverse(p.send_index[me]))
        return ops.combine(y_slot, g["slot_row"], x.dtype)


def emulate(xs, w_gate, w1, w3, w2, owner, time_experts: bool = False):
    """N ranks of the expert-parallel layer on one GPU (xs: one token batch per rank).

    All ranks' grouped rows share one device buffer, so dispatch and return
    are row gathers (``moe_gather_rows``). Returns (ys, plan, per-rank expert
    milliseconds or None).
    """
    import torch
    ops = CudaOps()
    E = len(owner)
    owner = _as_placement(owner, E)
    N = 1 + max(q for reps in owner for q in reps)
    groups = [ops.route_and_group(x, w_gate, E) for x in xs]
    p = plan(np.stack([g["counts"].cpu().numpy() for g in groups]), owner)
    base = np.cumsum([0] + [g["x_perm"].shape[0] for g in groups])
    all_rows = torch.cat([g["x_perm"] for g in groups])
    all_w = _gate_rows(torch.cat([g["perm_w"] for g in groups]))
    # receive buffer of q (source after source) composed with q's regroup
    y_parts, spans, ms = [], [], []
    for q in range(N):
        recv_global = np.concatenate(
            [base[s] + p.send_index[s][p.send_splits[s, :q].sum():p.send_splits[s, :q + 1].sum()] for s in range(N)])
        g_idx = recv_global[p.regroup[q]]
        rows = ops.gather(all_rows, g_idx)
        gate = ops.gather(all_w, g_idx)[:, 0].contiguous()
        ex = p.experts[q]
        wl = tuple(w[ex].contiguous() for w in (w1, w3, w2))
        if time_experts:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
        y_parts.append(ops.experts(rows, p.local_offsets[q], gate, *wl))
        if time_experts:
            b.record()
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        spans.append(g_idx)
    # return: row j of the stacked expert outputs came from global row spans[..][j]
    y_all = torch.cat(y_parts)
    src_of = np.concatenate(spans)
    ys = []
    for s, g in enumerate(groups):
        n = g["x_perm"].shape[0]
        where = np.full(n, -1, dtype=np.int64)
        mine = (src_of >= base[s]) & (src_of < base[s] + n)
        where[src_of[mine] - base[s]] = np.nonzero(mine)[0]
        y_slot = ops.gather(y_all, where) if n else y_all[:0]
        ys.append(ops.combine(y_slot, g["slot_row"], xs[s].dtype))
    return ys, p, (ms if time_experts else None)
