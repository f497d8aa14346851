"""The expert-parallel partition of the path (backward_token_expert_gb300.
expert_shard) with the library's kernels doing every step's arithmetic.

Two or three processes share the one GPU; each holds a block of tokens and
owns a block of experts, and they exchange over gloo on CPU tensors only, so
no kernel of one process ever waits on another process.  Each rank runs,
through the C ABI: route statistics on its tokens (the routed counts and
gate-probability sums are then all-reduced), scores of its pairs, selection
over all candidates of its experts (received from every rank), compaction of
the rows the expert owners ask of it, and the grouped GEMMs on its experts'
segments.  The union over ranks must equal the single-process GPU step bit
for bit (counts, quotas, selection, compacted rows, dW and the input-gradient
rows: each expert's rows arrive in the same order, so its products accumulate
in the same order), and the fp64 oracle where the parity tests compare with
it."""

import os
import socket
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
from gpu_common import SCORE_RTOL, bf16_np, built_library, custom_inputs, need_gpu, rel_close
from workloads import generate, get_workload

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": lambda: generate(get_workload("tiny_T256_E8_k2_h64_I32")),
    # odd expert count, k = 3, dead experts, experts over capacity
    "ragged": lambda: custom_inputs(T=600, E=13, k=3, h=48, I=40, s=1.4, rho=Fraction(1, 2), seed=5, dead=2),
    # several 256-wide tiles per expert and K blocks with ragged tails
    "tiles": lambda: custom_inputs(T=4096, E=16, k=4, h=512, I=320, s=0.8, rho=Fraction(3, 4), seed=11),
}


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    built_library()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _bf16(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _rank_path(rank, world, case, X):
    import torch

    from backward_token_expert_gb300 import lrm as L
    from backward_token_expert_gb300.pipeline import Recalibration

    inp = CASES[case]()
    w = inp.workload
    plan = X.ShardPlan(w.T, w.E, w.k, world, rank)
    t0, t1 = plan.token_range()
    p0, p1 = plan.pair_range()
    e0, e1 = plan.expert_range()
    Tl, El = t1 - t0, e1 - e0
    g, phi = _bf16(inp.g[t0:t1]), _bf16(inp.phi[p0:p1])
    alpha = torch.from_numpy(inp.alpha[p0:p1]).cuda()
    logits = torch.from_numpy(inp.logits[t0:t1]).cuda()
    idx_np = inp.expert_idx[t0:t1]
    idx = torch.from_numpy(idx_np).cuda()
    rec = Recalibration(Tl, w.E, w.k, w.h, w.I, w.cf, w.rho)
    try:
        # 1. routing statistics of this rank's tokens, then the global counts
        rec.route_stats(logits, idx)
        torch.cuda.synchronize()
        local_counts = rec.buf.counts.cpu().numpy().astype(np.int64)
        assert np.array_equal(local_counts, np.bincount(idx_np.reshape(-1), minlength=w.E))
        psum_local = torch.from_numpy(rec.buf.P.cpu().numpy().astype(np.float64) * Tl)
        counts, psum = X.global_route_counts(plan, torch.from_numpy(idx_np.astype(np.int64)), psum_local)
        counts = counts.numpy()
        C, quota = O.capacity_and_quotas(counts, w.N, w.E, w.cf, w.rho)

        # 2. scores of this rank's pairs; candidates to the expert owners
        rec.score(g, phi, alpha)
        torch.cuda.synchronize()
        R_local = rec.buf.score[: p1 - p0].cpu()
        cand = X.exchange_candidates(plan, R_local, torch.from_numpy(idx_np.astype(np.int64)))

        # 3. selection over all candidates of the owned experts: the received
        # candidates, grouped by expert in ascending pair id, are the bucket of
        # a layer of n_cand pairs and El experts
        order = np.lexsort((cand.u.numpy(), cand.e.numpy()))
        cu = cand.u.numpy()[order]
        ce = cand.e.numpy()[order] - e0
        n_cand = len(cu)
        own_q = quota[e0:e1].astype(np.int32)
        total = int(own_q.sum())
        so_own = np.zeros(El + 1, dtype=np.int64)
        so_own[1:] = np.cumsum(own_q)
        if total:
            dims_sel = L.dims_of(n_cand, El, 1, w.h, w.I)
            score_c = torch.from_numpy(cand.R.numpy()[order].astype(np.float32)).cuda()
            offs = np.zeros(El + 1, dtype=np.int32)
            offs[1:] = np.cumsum(np.bincount(ce, minlength=El))
            offsets = torch.from_numpy(offs).cuda()
            bucket = torch.arange(n_cand, dtype=torch.int32, device="cuda")
            q_dev = torch.from_numpy(own_q).cuda()
            sel_off = torch.zeros(El + 1, dtype=torch.int32, device="cuda")
            sel_ids = torch.zeros(total, dtype=torch.int32, device="cuda")
            ws_bytes = max(256, L.lrm_workspace_size(rec.ctx, L.LRM_OP_SELECT, dims_sel))
            ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
            L.lrm_select(rec.ctx, score_c, offsets, bucket, q_dev, dims_sel, total, sel_off, sel_ids, ws, ws_bytes)
            torch.cuda.synchronize()
            assert np.array_equal(sel_off.cpu().numpy(), so_own)
            sel_u = torch.from_numpy(cu[sel_ids.cpu().numpy().astype(np.int64)])
        else:
            sel_u = torch.zeros(0, dtype=torch.int64)

        # 4./5. requests to the token owners; they compact the asked rows
        req = X.request_rows(plan, sel_u)
        asked = req.asked_u.numpy() - p0
        n_req = len(asked)
        rows = torch.zeros((n_req, w.h + w.I), dtype=torch.int16)
        if n_req:
            # the asked rows as one segment (row offsets [0, n_req, ..., n_req])
            dims_c = L.dims_of(Tl, w.E, w.k, w.h, w.I)
            dc = torch.empty(n_req, w.h, dtype=torch.bfloat16, device="cuda")
            pc = torch.empty(n_req, w.I, dtype=torch.bfloat16, device="cuda")
            off_c = torch.tensor([0] + [n_req] * w.E, dtype=torch.int32, device="cuda")
            ids_c = torch.from_numpy(asked.astype(np.int32)).cuda()
            L.lrm_compact(rec.ctx, g, phi, alpha, off_c, ids_c, dims_c, n_req, dc, pc)
            torch.cuda.synchronize()
            rows = torch.cat([dc.view(torch.int16), pc.view(torch.int16)], dim=1).cpu()
        got = X.send_rows(req, rows)
        delta_c = got[:, : w.h].contiguous().view(torch.bfloat16)
        phi_c = got[:, w.h:].contiguous().view(torch.bfloat16)

        # 6. grouped GEMMs on the owned experts' segments
        dims_g = L.dims_of(max(1, n_cand), El, 1, w.h, w.I)
        W_own = _bf16(inp.W[e0:e1])
        so_dev = torch.from_numpy(so_own.astype(np.int32)).cuda()
        dW = torch.full((El, w.h, w.I), 7.0, dtype=torch.float32, device="cuda")
        dphi = torch.zeros((max(1, total), w.I), dtype=torch.bfloat16, device="cuda")
        dc_dev = delta_c.cuda() if total else torch.zeros((1, w.h), dtype=torch.bfloat16, device="cuda")
        pc_dev = phi_c.cuda() if total else torch.zeros((1, w.I), dtype=torch.bfloat16, device="cuda")
        L.lrm_grouped_dgrad(rec.ctx, dc_dev, W_own, so_dev, dims_g, total, dphi)
        L.lrm_grouped_wgrad(rec.ctx, dc_dev, pc_dev, so_dev, dims_g, total, 0, dW)
        torch.cuda.synchronize()
        assert rec.device_status() == 0
        dphi_rows = dphi[:total].view(torch.int16).cpu()

        # 7. input-gradient rows back to the token owners, at their pairs' rows
        back = X.return_rows(req, dphi_rows).numpy()
        local = np.zeros((p1 - p0, w.I), dtype=np.int16)
        local[asked] = back
        return dict(counts=counts, psum=psum.numpy(), quota=quota, C=C, R=R_local.numpy(), so=so_own,
                    sel_u=sel_u.numpy(), delta_c=got[:, : w.h].numpy(), phi_c=got[:, w.h:].numpy(),
                    dW=dW.cpu().numpy(), dphi_local=local, p0=p0, p1=p1, experts=(e0, e1))
    finally:
        rec.close()


def _worker(rank, world, port, case, q):
    import torch.distributed as dist

    from backward_token_expert_gb300 import expert_shard as X

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, _rank_path(rank, world, case, X)))
    except Exception as ex:  # report at once instead of leaving the parent waiting
        q.put((rank, f"{type(ex).__name__}: {ex}"))
        raise
    finally:
        dist.destroy_process_group()


def _run(case, world):
    import multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, case, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    try:
        for _ in range(world):
            rank, out = q.get(timeout=300)
            assert not isinstance(out, str), f"rank {rank}: {out}"
            res[rank] = out
    finally:
        for p in procs:
            p.join(timeout=120)
    for p in procs:
        assert p.exitcode == 0
    return res


def _single_process(inp):
    """The same layer as one process runs it (the reference for bit equality)."""
    import torch

    from backward_token_expert_gb300.pipeline import Recalibration, to_device_inputs

    w = inp.workload
    rec = Recalibration(w.T, w.E, w.k, w.h, w.I, w.cf, w.rho)
    try:
        d = to_device_inputs(inp)
        rec.run(d["logits"], d["expert_idx"], d["g"], d["phi"], d["alpha"], d["W"])
        torch.cuda.synchronize()
        b = rec.buf
        so = b.sel_offsets.cpu().numpy().astype(np.int64)
        tot = int(so[-1])
        return dict(counts=b.counts.cpu().numpy(), quota=b.quota.cpu().numpy(), P=b.P.cpu().numpy(),
                    score=b.score.cpu().numpy()[: w.N], so=so, ids=b.sel_ids.cpu().numpy()[:tot].astype(np.int64),
                    delta_c=bf16_np(b.delta_c[:tot]), phi_c=bf16_np(b.phi_c[:tot]),
                    dphi=b.dphi_c[:tot].view(torch.int16).cpu().numpy(), dW=b.dW.cpu().numpy(),
                    flags=rec.device_status())
    finally:
        rec.close()


@pytest.mark.parametrize("case,world", [("tiny", 2), ("ragged", 2), ("ragged", 3), ("tiles", 2)])
def test_expert_sharded_kernels_equal_single_process(case, world):
    inp = CASES[case]()
    w = inp.workload
    res = _run(case, world)
    ref = _single_process(inp)
    assert ref["flags"] == 0
    st = O.route_stats(inp.logits, inp.expert_idx, w.E, w.cf, w.rho)
    # scores: every rank's are the single-process ones (one token per warp either way)
    R = np.concatenate([res[r]["R"] for r in range(world)])
    assert np.array_equal(R.view(np.uint32), ref["score"].view(np.uint32))
    R64 = O.score(inp.g, inp.phi, inp.alpha, w.k)
    assert np.all(rel_close(R, R64, SCORE_RTOL, 1e-30))
    # the oracle's selection on these fp32 scores
    so_o, ids_o = O.select(R.astype(np.float64), inp.expert_idx, w.E, st["quota"])
    assert np.array_equal(ids_o, ref["ids"])
    union_u, union_dc, union_pc, union_dphi = [], [], [], []
    dW = np.zeros((w.E, w.h, w.I), dtype=np.float32)
    dphi_scatter = np.zeros((w.N, w.I), dtype=np.int16)
    for r in range(world):
        out = res[r]
        assert np.array_equal(out["counts"], st["counts"]) and np.array_equal(out["counts"], ref["counts"])
        assert np.allclose(out["psum"] / w.T, st["P"], rtol=1e-5, atol=1e-9)
        assert out["C"] == st["C"] and np.array_equal(out["quota"], ref["quota"])
        e0, e1 = out["experts"]
        dW[e0:e1] = out["dW"]
        for i, e in enumerate(range(e0, e1)):
            a, b = out["so"][i], out["so"][i + 1]
            union_u.append(out["sel_u"][a:b])
            union_dc.append(out["delta_c"][a:b])
            union_pc.append(out["phi_c"][a:b])
        dphi_scatter[out["p0"]:out["p1"]] = out["dphi_local"]
    assert np.array_equal(np.concatenate(union_u), ref["ids"])
    assert np.array_equal(np.concatenate(union_dc).view(np.uint16), ref["delta_c"])
    assert np.array_equal(np.concatenate(union_pc).view(np.uint16), ref["phi_c"])
    dc_o, pc_o, _ = O.compact(inp.g, inp.phi, inp.alpha, ref["ids"], w.k)
    assert np.array_equal(ref["delta_c"], dc_o) and np.array_equal(ref["phi_c"], pc_o)
    # the GEMMs: bit for bit the single-process results
    assert np.array_equal(dW.view(np.uint32), ref["dW"].view(np.uint32))
    expect = np.zeros((w.N, w.I), dtype=np.int16)
    expect[ref["ids"]] = ref["dphi"]
    assert np.array_equal(dphi_scatter, expect)
