"""Expert parallelism: the host plan and the distributed forward over gloo ranks on CPU.

The per-rank steps (routing, grouping, row moves, experts, combine) run on CPU
stand-ins built from the fp64 oracle here, so that the exchange logic is
checked without a GPU: every rank's output must equal the single-process
oracle layer on its own tokens.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from sparse_mixture_experts_53_b300 import ep


def _counts(rng, N, E, T, skew=False):
    c = np.zeros((N, E), dtype=np.int64)
    for s in range(N):
        p = np.ones(E)
        if skew:
            p[:2] = 6.0
        p = p / p.sum()
        for _ in range(T):
            a, b = rng.choice(E, size=2, replace=False, p=p)
            c[s, a] += 1
            c[s, b] += 1
    return c


@pytest.mark.parametrize("N", [1, 2, 4, 8])
@pytest.mark.parametrize("balanced", [False, True])
def test_plan_moves_every_row_once_to_its_owner(N, balanced):
    rng = np.random.default_rng(N)
    counts = _counts(rng, N, 8, 37, skew=True)
    owner = ep.balanced_owners(counts.sum(0), N) if balanced else ep.contiguous_owners(8, N)
    p = ep.plan(counts, owner)
    assert np.array_equal(p.recv_splits, p.send_splits.T)
    # label every source row by (source, expert, rank in group), move labels as the plan says
    labels = []
    for s in range(N):
        lab = [(s, e, i) for e in range(8) for i in range(counts[s, e])]
        assert len(p.send_index[s]) == len(lab) and sorted(p.send_index[s]) == list(range(len(lab)))
        sent = [lab[j] for j in p.send_index[s]]
        cuts = np.cumsum([0] + p.send_splits[s].tolist())
        labels.append([sent[cuts[q]:cuts[q + 1]] for q in range(N)])
    seen = set()
    for q in range(N):
        recv = [r for s in range(N) for r in labels[s][q]]
        assert sorted(p.regroup[q]) == list(range(len(recv)))
        local = [recv[j] for j in p.regroup[q]]
        for j, e in enumerate(p.experts[q]):
            grp = local[p.local_offsets[q][j]:p.local_offsets[q][j + 1]]
            assert all(lab[1] == e for lab in grp)
            assert grp == sorted(grp)  # sources in order, then the source's own order
        assert all(owner[lab[1]] == q for lab in local)
        seen.update(local)
    assert len(seen) == int(counts.sum())
    assert np.array_equal(p.rows_per_rank, [counts[:, p.experts[q]].sum() for q in range(N)])


def test_balanced_placement():
    load = np.array([600, 380, 10, 50, 250, 70, 13, 0])
    own = ep.balanced_owners(load, 4)
    assert np.all(np.bincount(own, minlength=4) == 2)
    per = np.bincount(own, weights=load, minlength=4)
    assert per.max() == 600  # the hottest expert alone; the contiguous placement gives 980
    assert np.bincount(ep.contiguous_owners(8, 4), weights=load, minlength=4).max() == 980


@pytest.mark.parametrize("N,slots", [(2, 5), (4, 3), (8, 2), (8, 4)])
def test_plan_with_replicas_splits_each_block_over_its_copies(N, slots):
    rng = np.random.default_rng(100 + N)
    counts = _counts(rng, N, 8, 53, skew=True)
    place = ep.replicated_placement(counts.sum(0), N, slots)
    assert all(len(set(r)) == len(r) for r in place)
    assert max(sum(q in r for r in place) for q in range(N)) <= slots
    # on two ranks the single-copy placement already splits the two hot experts
    assert any(len(r) > 1 for r in place) == (N > 2)
    p = ep.plan(counts, place)
    assert np.array_equal(p.recv_splits, p.send_splits.T)
    labels = []
    for s in range(N):
        lab = [(s, e, i) for e in range(8) for i in range(counts[s, e])]
        assert sorted(p.send_index[s]) == list(range(len(lab)))
        sent = [lab[j] for j in p.send_index[s]]
        cuts = np.cumsum([0] + p.send_splits[s].tolist())
        labels.append([sent[cuts[q]:cuts[q + 1]] for q in range(N)])
    got = {}
    for q in range(N):
        recv = [r for s in range(N) for r in labels[s][q]]
        local = [recv[j] for j in p.regroup[q]]
        for j, e in enumerate(p.experts[q]):
            grp = local[p.local_offsets[q][j]:p.local_offsets[q][j + 1]]
            assert all(lab[1] == e for lab in grp) and grp == sorted(grp)
            for lab in grp:
                assert lab not in got
                got[lab] = q
    assert len(got) == int(counts.sum())
    # source s's rows of e: consecutive chunks, in the order of e's copies, sizes within one
    for s in range(N):
        for e in range(8):
            dest = [got[(s, e, i)] for i in range(counts[s, e])]
            k = len(place[e])
            want = [place[e][j] for j in range(k) for _ in range((counts[s, e] * (j + 1)) // k - (counts[s, e] * j) // k)]
            assert dest == want


def test_replicated_placement_spreads_a_hot_expert():
    # one expert takes 40% of the rows: on 8 ranks it alone bounds the step
    load = np.array([3200, 700, 700, 700, 700, 700, 700, 600])
    own = ep.balanced_owners(load, 8)
    assert np.bincount(own, weights=load, minlength=8).max() == 3200
    place = ep.replicated_placement(load, 8, 2)
    per = np.zeros(8)
    for e, r in enumerate(place):
        for q in r:
            per[q] += load[e] / len(r)
    assert per.max() <= 0.5 * 3200 and per.sum() == load.sum()
    assert len(place[0]) >= 4
    # a flat load gains nothing from copies, so none are made
    flat = ep.replicated_placement(np.full(8, 100), 4, 4)
    assert all(len(r) == 1 for r in flat)


class CpuOps:
    """fp64 stand-ins of the per-rank kernels, from the oracle (test infrastructure)."""

    def route_and_group(self, x, w_gate, E):
        X = x.numpy()
        l = oracle.router_logits(X, w_gate.numpy())
        idx, g, _ = oracle.top_k_gates(l, 2)
        p = oracle.permute(idx, g, E)
        return dict(counts=torch.from_numpy(p["counts"]), slot_row=torch.from_numpy(p["slot_row"]),
                    perm_w=torch.from_numpy(p["perm_w"]), x_perm=torch.from_numpy(X[p["perm_token"]]))

    def gather(self, src, index):
        return src[torch.as_tensor(np.asarray(index, dtype=np.int64))]

    def experts(self, rows, local_offsets, gate, w1, w3, w2):
        return torch.from_numpy(oracle.expert_ffn_slots(rows.numpy(), local_offsets, gate.numpy(), w1.numpy(),
                                                        w3.numpy(), w2.numpy()))

    def combine(self, y_slot, slot_row, dtype):
        return torch.from_numpy(oracle.combine(y_slot.numpy(), slot_row.numpy()))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _layer(seed, T, d=16, ffn=8, E=8, skew=False):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    wg = rng.standard_normal((E, d)) / np.sqrt(d)
    if skew:
        wg[:2] += 0.8 * np.sign(x.mean(0))
    w1 = rng.standard_normal((E, ffn, d)) / np.sqrt(d)
    w3 = rng.standard_normal((E, ffn, d)) / np.sqrt(d)
    w2 = rng.standard_normal((E, d, ffn)) / np.sqrt(ffn)
    return x, wg, w1, w3, w2


def _rank(rank, world, port, mode, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x_all, wg, w1, w3, w2 = _layer(11, 24 * world, skew=True)
        x = x_all[24 * rank:24 * (rank + 1)]
        # every rank derives the same placement from the whole batch's routing
        l = oracle.router_logits(x_all, wg)
        idx, _, _ = oracle.top_k_gates(l, 2)
        load = np.bincount(idx.ravel(), minlength=8)
        if mode == "replicated":
            # copies of two hot experts (a load heavier than this small batch's)
            owner = ep.replicated_placement(np.array([900, 700, 50, 50, 50, 50, 50, 50]), world, 8 // world + 1)
            assert any(len(r) > 1 for r in owner)
            mine = [e for e in range(8) if rank in owner[e]]
        else:
            owner = ep.balanced_owners(load, world) if mode == "balanced" else ep.contiguous_owners(8, world)
            mine = [e for e in range(8) if owner[e] == rank]
        layer = ep.ExpertParallelLayer(torch.from_numpy(wg), torch.from_numpy(w1[mine]), torch.from_numpy(w3[mine]),
                                       torch.from_numpy(w2[mine]), owner, ops=CpuOps())
        y = layer.forward(torch.from_numpy(x)).numpy()
        ref = oracle.layer_forward(x, wg, w1, w3, w2)["y"]
        out.put((rank, float(np.max(np.abs(y - ref))), layer.last_plan.rows_per_rank.tolist()))
    except Exception as e:  # report instead of leaving the parent waiting
        out.put((rank, float("inf"), repr(e)))
        raise
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(180)
@pytest.mark.parametrize("world,mode", [(2, "contiguous"), (4, "contiguous"), (4, "balanced"), (4, "replicated")])
def test_distributed_forward_equals_the_single_process_layer(world, mode):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, mode, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=150) for _ in range(world))
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for rank, err, rows in res:
        assert err <= 1e-12, (rank, err)
    assert sum(res[0][2]) == 2 * 24 * world  # every slot of every rank ran once
