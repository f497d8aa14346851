"""The inverse mapping (LRMoE Alg. 1, ScatterWithZeros; sec. 3.4) on the
GPU: the scattered input gradient holds, at row u of every retained pair, the
same bits as the compacted dgrad output, and exact zeros at every other row;
against the oracle it is the scattered fp64 gradient within the GEMM bound."""

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
from gpu_common import bf16_np, built_library, custom_inputs, need_gpu
from workloads import generate

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    built_library()


def _scatter_check(inp, quota=None):
    from backward_token_expert_gb300.pipeline import Recalibration, to_device_inputs

    w = inp.workload
    rec = Recalibration(w.T, w.E, w.k, w.h, w.I, w.cf, w.rho, max_rows=w.N if quota is not None else None)
    try:
        d = to_device_inputs(inp)
        q = None if quota is None else torch.as_tensor(np.asarray(quota, dtype=np.int32), device="cuda")
        rec.route_stats(d["logits"], d["expert_idx"], quota_override=q)
        rec.backward_steps(d["g"], d["phi"], d["alpha"], d["W"])
        # rows nobody writes would keep these NaN bits
        rows = torch.full((w.N, w.I), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        rec.dgrad_scatter(d["W"], rows)
        torch.cuda.synchronize()
        assert rec.device_status() == 0
        b = rec.buf
        so = b.sel_offsets.cpu().numpy().astype(np.int64)
        ids = b.sel_ids.cpu().numpy()[: so[-1]].astype(np.int64)
        compact = bf16_np(b.dphi_c[: so[-1]])
        out = bf16_np(rows)
    finally:
        rec.close()
    kept = np.zeros(w.N, dtype=bool)
    kept[ids] = True
    assert np.array_equal(out[ids], compact)
    assert np.all(out[~kept] == 0)
    # against the oracle: the scattered fp64 input gradient
    dphi = O.grouped_dgrad(inp.g, inp.W, inp.alpha, so, ids, w.E, w.k)
    ref = O.scatter_with_zeros(np.concatenate([dphi[e] for e in range(w.E)], axis=0), ids, w.N)
    got = O.bf16_to_f64(out)
    for e in range(w.E):
        seg = ids[so[e]:so[e + 1]]
        if seg.size:
            assert np.linalg.norm(got[seg] - ref[seg]) <= 5e-3 * np.linalg.norm(ref[seg])
    return kept


def test_scatter_tiny_workload():
    kept = _scatter_check(generate("tiny_T256_E8_k2_h64_I32"))
    assert 0 < kept.sum() < kept.size


def test_scatter_ragged_sizes_and_empty_experts():
    inp = custom_inputs(T=3000, E=12, k=3, h=192, I=200, s=1.6, rho=Fraction(1, 2), seed=31, dead=2)
    _scatter_check(inp)


def test_scatter_with_caller_quotas_keeping_nothing_and_everything():
    inp = custom_inputs(T=640, E=8, k=2, h=64, I=64, s=0.8, seed=32)
    n = np.bincount(inp.expert_idx.reshape(-1), minlength=8)
    quota = n.copy()
    quota[0] = 0
    quota[2:] = np.maximum(n[2:] - 1, 0)
    _scatter_check(inp, quota=quota)


def test_scatter_full_retention_writes_every_row():
    inp = custom_inputs(T=1024, E=8, k=2, h=128, I=96, s=0.3, rho=Fraction(1), seed=33)
    w = inp.workload
    inp = type(inp)(**{**inp.__dict__, "workload": type(w)(**{**w.__dict__, "cf": Fraction(8)})})
    kept = _scatter_check(inp)
    assert kept.all()
