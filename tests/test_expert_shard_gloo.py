"""The expert-parallel partition of the path (backward_token_expert_gb300.
expert_shard) on CPU ranks with the gloo backend.

Each rank holds a block of tokens and owns a block of experts.  The ranks run
the path with the fp64 oracle for the arithmetic and the module's exchanges
between the steps: the all-reduce of the routed counts and summed gate
probabilities, the candidates (u, e, R) to the expert owner, selection there,
the requests back to the token owners, the compacted rows to the expert
owner, the grouped GEMMs there, and the input-gradient rows back to the
token owners.  The union over ranks must equal the single-process oracle:
counts, quotas, selection and compacted rows bit for bit, the gradients to
the last bits of fp64 (the same rows in the same order), the importance
within fp64 rounding of a different summation order.
"""

import os
import socket
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
from workloads import generate, get_workload

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(case):
    from gpu_common import custom_inputs

    if case == "tiny":
        return generate(get_workload("tiny_T256_E8_k2_h64_I32"))
    # odd expert count, k = 3, two dead experts, many experts over capacity
    return custom_inputs(T=600, E=13, k=3, h=48, I=40, s=1.4, rho=Fraction(1, 2), seed=5, dead=2)


def _worker(rank, world, port, case, q):
    import torch.distributed as dist

    from backward_token_expert_gb300 import expert_shard as X

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        _rank_path(rank, world, case, q, X)
    except Exception as ex:  # report at once instead of leaving the parent waiting
        q.put((rank, f"{type(ex).__name__}: {ex}"))
        raise
    finally:
        dist.destroy_process_group()


def _rank_path(rank, world, case, q, X):
    inp = _inputs(case)
    w = inp.workload
    plan = X.ShardPlan(w.T, w.E, w.k, world, rank)
    t0, t1 = plan.token_range()
    p0, p1 = plan.pair_range()
    e0, e1 = plan.expert_range()
    g, phi, alpha = inp.g[t0:t1], inp.phi[p0:p1], inp.alpha[p0:p1]
    idx = torch.from_numpy(inp.expert_idx[t0:t1].astype(np.int64))

    # 1. routing statistics from the global counts
    psum = torch.from_numpy(O.softmax_rows(inp.logits[t0:t1]).sum(axis=0))
    counts, psum = X.global_route_counts(plan, idx, psum)
    counts = counts.numpy()
    C, quota = O.capacity_and_quotas(counts, w.N, w.E, w.cf, w.rho)

    # 2. scores at the token owner, candidates to the expert owner
    R = O.score(g, phi, alpha, w.k)
    cand = X.exchange_candidates(plan, torch.from_numpy(R), idx)
    # 3. selection over all candidates of the owned experts
    own_q = np.where((np.arange(w.E) >= e0) & (np.arange(w.E) < e1), quota, 0)
    so, pick = O.select(cand.R.numpy(), cand.e.numpy(), w.E, own_q)
    sel_u = cand.u[torch.from_numpy(pick)]

    # 4./5. requests to the token owners, compacted rows back to the owner
    req = X.request_rows(plan, sel_u)
    dc, pc, _ = O.compact(g, phi, alpha, req.asked_u.numpy() - p0, w.k)
    rows = torch.from_numpy(np.concatenate([dc, pc], axis=1).view(np.int16))
    got = X.send_rows(req, rows).numpy().view(np.uint16)
    delta_c, phi_c = got[:, :w.h], got[:, w.h:]

    # 6. GEMMs on the owned experts' segments
    owned = range(e0, e1)
    dW = O.grouped_wgrad_from_compact(delta_c, phi_c, so, w.E, owned)
    dphi = O.grouped_dgrad_from_compact(delta_c, inp.W, so, w.E, owned)
    dphi_rows = np.concatenate([dphi[e] for e in owned], axis=0) if so[-1] else np.zeros((0, w.I))
    # 7. input-gradient rows back to the token owners, at their pairs' rows
    back = X.return_rows(req, torch.from_numpy(dphi_rows)).numpy()
    local = np.zeros((p1 - p0, w.I))
    local[req.asked_u.numpy() - p0] = back

    q.put((rank, dict(counts=counts, psum=psum.numpy(), quota=quota, C=C, so=so, sel_u=sel_u.numpy(),
                      delta_c=delta_c, phi_c=phi_c, dW={e: dW[e] for e in owned}, dphi_local=local,
                      p0=p0, p1=p1, experts=(e0, e1))))


def _run(case, world):
    import multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, case, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        rank, out = q.get(timeout=180)
        assert not isinstance(out, str), f"rank {rank}: {out}"
        res[rank] = out
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return res


@pytest.mark.parametrize("case,world", [("tiny", 2), ("ragged", 2), ("ragged", 3)])
def test_expert_sharded_path_equals_single_process(case, world):
    inp = _inputs(case)
    w = inp.workload
    res = _run(case, world)
    ref = O.backward_recalibration(inp)
    st, so, ids = ref["stats"], ref["sel_offsets"], ref["sel_ids"]
    ref_dW = O.grouped_wgrad_from_compact(ref["delta_c"], ref["phi_c"], so, w.E)
    ref_dphi = O.grouped_dgrad_from_compact(ref["delta_c"], inp.W, so, w.E)
    dphi_rows = np.concatenate([ref_dphi[e] for e in range(w.E)], axis=0)
    ref_scatter = O.scatter_with_zeros(dphi_rows, ids, w.N)
    union_u, union_dc, union_pc = [], [], []
    for r in range(world):
        out = res[r]
        assert np.array_equal(out["counts"], st["counts"])
        assert np.allclose(out["psum"] / w.T, st["P"], rtol=1e-12, atol=0)
        assert out["C"] == st["C"] and np.array_equal(out["quota"], st["quota"])
        e0, e1 = out["experts"]
        for e in range(e0, e1):
            a, b = out["so"][e], out["so"][e + 1]
            union_u.append(out["sel_u"][a:b])
            union_dc.append(out["delta_c"][a:b])
            union_pc.append(out["phi_c"][a:b])
            assert np.allclose(out["dW"][e], ref_dW[e], rtol=1e-12, atol=1e-300)
        # the inverse mapping of this rank's pairs: retained rows, zeros elsewhere
        assert np.allclose(out["dphi_local"], ref_scatter[out["p0"]:out["p1"]], rtol=1e-12, atol=1e-300)
    assert np.array_equal(np.concatenate(union_u), ids)  # expert-major, ascending u within an expert
    assert np.array_equal(np.concatenate(union_dc), ref["delta_c"])
    assert np.array_equal(np.concatenate(union_pc), ref["phi_c"])
    assert sum(len(x) for x in union_u) == st["retained"]


def test_plan_blocks_cover_experts_and_tokens():
    from backward_token_expert_gb300.expert_shard import ShardPlan

    for T, E, k, world in ((256, 8, 2, 2), (1000, 13, 3, 3), (7, 5, 1, 4)):
        plans = [ShardPlan(T, E, k, world, r) for r in range(world)]
        assert [p.expert_range()[0] for p in plans] + [E] == [0] + [p.expert_range()[1] for p in plans]
        assert [p.token_range()[0] for p in plans] + [T] == [0] + [p.token_range()[1] for p in plans]
        e = torch.arange(E)
        owner = plans[0].expert_owner(e)
        for r, p in enumerate(plans):
            lo, hi = p.expert_range()
            assert torch.all(owner[lo:hi] == r)
            u = torch.arange(*p.pair_range())
            assert torch.all(p.token_owner_of_pair(u) == r)
