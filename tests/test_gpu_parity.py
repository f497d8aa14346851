"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Integer work (counts, offsets, bucket, quotas, selected ids, compacted rows)
must match bit for bit; scores within 1e-5 relative; GEMM outputs within
5e-3 relative Frobenius error per expert.  Selection is compared with the
oracle rerun on the GPU's fp32 scores (ties to the lower pair index).
"""

from fractions import Fraction

import numpy as np
import pytest

import oracle as O
from gpu_common import (
    SCORE_RTOL,
    built_library,
    check_compaction,
    check_gemms,
    check_route_stats,
    check_selection,
    custom_inputs,
    need_gpu,
    rel_close,
    run_gpu,
)
from workloads import generate

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    built_library()


def full_check(inp, quota=None, padded=False):
    w = inp.workload
    st = O.route_stats(inp.logits, inp.expert_idx, w.E, w.cf, w.rho, quota=quota)
    gpu = run_gpu(inp, quota=quota, padded=padded)
    if quota is None:
        check_route_stats(gpu, inp, st)
        assert np.array_equal(gpu["quota"], st["quota"])
        assert gpu["summary"]["retained"] == st["retained"]
    else:
        assert gpu["flags"] == 0
        assert np.array_equal(gpu["counts"], st["counts"])
    R = O.score(inp.g, inp.phi, inp.alpha, w.k)
    assert np.all(rel_close(gpu["score"], R, SCORE_RTOL, 1e-30))
    so, ids = check_selection(gpu, inp, st["quota"])
    check_compaction(gpu, inp, ids)
    check_gemms(gpu, inp, so, ids)
    return gpu, st, so, ids


def test_tiny_workload_whole_path():
    full_check(generate("tiny_T256_E8_k2_h64_I32"))


def test_ragged_sizes_span_several_tiles():
    # h = 320 (K tail of 0 in 64s, M tail of 64 rows), I = 200 (N tail), many experts
    full_check(custom_inputs(T=1536, E=16, k=4, h=320, I=200, s=1.0, rho=Fraction(3, 4), seed=1))


def test_wide_expert_uses_256_column_tiles():
    full_check(custom_inputs(T=4096, E=8, k=2, h=256, I=768, s=0.5, rho=Fraction(1, 2), seed=2))


def test_rows_too_wide_for_the_staging_ring():
    # h + I = 17408: a g row and a phi row no longer fit two slots per warp of
    # the TMA-staged compaction, so the 128-bit copy kernel does it
    full_check(custom_inputs(T=192, E=4, k=2, h=16384, I=1024, s=0.5, rho=Fraction(3, 4), seed=7))


def test_non_power_of_two_experts_and_k():
    full_check(custom_inputs(T=999, E=20, k=6, h=136, I=1408, s=1.2, rho=Fraction(3, 5), seed=3,
                             phi_scale="lognormal"))


def test_empty_and_oversized_experts():
    inp = custom_inputs(T=3000, E=12, k=3, h=192, I=128, s=1.6, rho=Fraction(1, 2), seed=4, dead=2)
    w = inp.workload
    n = np.bincount(inp.expert_idx.reshape(-1), minlength=w.E)
    C = (w.cf.numerator * w.N) // (w.cf.denominator * w.E)
    assert (n == 0).sum() >= 2 and (n > C).sum() >= 1
    full_check(inp)


def test_caller_quotas_zero_and_full_and_fig4_pattern():
    inp = custom_inputs(T=640, E=8, k=2, h=64, I=64, s=0.8, seed=5)
    n = np.bincount(inp.expert_idx.reshape(-1), minlength=8)
    quota = n.copy()
    quota[0] = 0  # keep nothing
    quota[1] = n[1]  # keep everything
    quota[2:] = np.maximum(n[2:] - 1, 0)  # drop one per expert, as in LRMoE Fig. 4
    full_check(inp, quota=quota)


def test_all_equal_scores_keep_lowest_pair_indices():
    inp = custom_inputs(T=512, E=4, k=2, h=64, I=32, seed=6)
    inp.g[:] = inp.g[0]
    inp.phi[:] = inp.phi[0]
    inp.alpha[:] = np.float32(0.5)
    gpu, st, so, ids = full_check(inp)
    e_u = inp.expert_idx.reshape(-1)
    for e in range(4):
        cand = np.flatnonzero(e_u == e)
        assert np.array_equal(ids[so[e]:so[e + 1]], cand[: st["quota"][e]])


def test_many_exact_ties():
    inp = custom_inputs(T=2048, E=8, k=2, h=64, I=64, seed=7)
    rng = np.random.default_rng(7)
    # phi rows from four distinct rows -> scores take few distinct values per token
    inp.phi[:] = inp.phi[rng.integers(0, 4, size=inp.phi.shape[0])]
    inp.g[:] = inp.g[rng.integers(0, 3, size=inp.g.shape[0])]
    inp.alpha[:] = np.float32(0.5)
    full_check(inp)


def test_full_retention_is_dense_moe_backward():
    inp = custom_inputs(T=1024, E=8, k=2, h=128, I=96, s=0.3, rho=Fraction(1), seed=8)
    w = inp.workload
    # CF large enough that no expert is capped: quotas equal the routed counts
    gpu = run_gpu(inp, cf=Fraction(8))
    st = O.route_stats(inp.logits, inp.expert_idx, w.E, Fraction(8), Fraction(1))
    assert np.array_equal(gpu["quota"], st["counts"])
    so, ids = check_selection(gpu, inp, st["quota"])
    check_gemms(gpu, inp, so, ids)


def test_zero_masked_comparator_matches_compacted():
    inp = custom_inputs(T=2048, E=8, k=2, h=256, I=256, s=0.8, rho=Fraction(3, 4), seed=9)
    w = inp.workload
    gpu, st, so, ids = full_check(inp, padded=True)
    C = st["C"]
    dpad, ppad = O.compact_padded(gpu["delta_c"], gpu["phi_c"], so, w.E, C)
    assert np.array_equal(gpu["delta_pad"].reshape(w.E, C, w.h), dpad)
    assert np.array_equal(gpu["phi_pad"].reshape(w.E, C, w.I), ppad)
    assert np.array_equal(gpu["pad_offsets"], np.arange(w.E + 1) * C)
    for e in range(w.E):
        q = int(so[e + 1] - so[e])
        ref = gpu["dW"][e].astype(np.float64)
        if q == 0:
            assert np.all(gpu["dW_pad"][e] == 0)
            continue
        assert np.linalg.norm(gpu["dW_pad"][e] - ref) <= 1e-5 * np.linalg.norm(ref)
        a = O.bf16_to_f64(gpu["dphi_pad"][e * C:e * C + q])
        b = O.bf16_to_f64(gpu["dphi_c"][so[e]:so[e] + q])
        assert np.linalg.norm(a - b) <= 1e-2 * np.linalg.norm(b)
        assert np.all(gpu["dphi_pad"][e * C + q:(e + 1) * C] == 0)


def test_wgrad_accumulate_adds_into_dW():
    import torch

    from backward_token_expert_gb300.pipeline import Recalibration, to_device_inputs

    inp = custom_inputs(T=512, E=4, k=2, h=128, I=128, seed=10)
    w = inp.workload
    rec = Recalibration(w.T, w.E, w.k, w.h, w.I, w.cf, w.rho)
    try:
        d = to_device_inputs(inp)
        rec.run(d["logits"], d["expert_idx"], d["g"], d["phi"], d["alpha"], d["W"])
        first = rec.buf.dW.clone()
        rec.wgrad(accumulate=1)
        torch.cuda.synchronize()
        assert torch.allclose(rec.buf.dW, 2 * first, rtol=1e-6, atol=0)
        assert rec.device_status() == 0
    finally:
        rec.close()


def test_run_to_run_determinism():
    inp = custom_inputs(T=1500, E=16, k=4, h=128, I=64, s=1.0, seed=11)
    a = run_gpu(inp)
    b = run_gpu(inp)
    for key in ("bucket", "score", "sel_ids", "delta_c", "phi_c", "dphi_c"):
        assert np.array_equal(a[key], b[key]), key
    assert np.array_equal(a["dW"].view(np.uint32), b["dW"].view(np.uint32))


def test_empty_batch():
    inp = custom_inputs(T=64, E=8, k=2, h=64, I=32, seed=12)
    gpu = run_gpu(inp, rho=Fraction(0))
    assert gpu["flags"] == 0
    assert np.all(gpu["sel_offsets"] == 0)
    assert np.all(gpu["dW"] == 0)


@pytest.mark.parametrize("T,E,mode,seed", [(6000, 1, "equal", 13), (20000, 1, "equal", 14),
                                           (16384, 2, "few", 15), (30000, 4, "few", 16),
                                           (40000, 2, "spread", 17)])
def test_large_experts_sampled_bracket_and_fallback(T, E, mode, seed):
    """Experts with thousands of candidates go through the sampled bracket
    (and its fallback when the bracket holds too many keys, e.g. all equal)."""
    inp = custom_inputs(T=T, E=E, k=1, h=64, I=32, s=0.0, rho=Fraction(3, 4), seed=seed)
    rng = np.random.default_rng(seed)
    if mode == "equal":
        inp.g[:] = inp.g[0]
        inp.phi[:] = inp.phi[0]
        inp.alpha[:] = np.float32(0.5)
    elif mode == "few":
        inp.phi[:] = inp.phi[rng.integers(0, 5, size=inp.phi.shape[0])]
        inp.g[:] = inp.g[rng.integers(0, 3, size=inp.g.shape[0])]
        inp.alpha[:] = np.float32(0.25)
    full_check(inp)


@pytest.mark.parametrize("T,E,k,h,I,rho", [(1, 1, 1, 8, 8, Fraction(1)), (3, 4, 4, 16, 8, Fraction(3, 4)),
                                           (100, 2, 2, 8, 8, Fraction(1, 2)), (300, 32, 32, 64, 40, Fraction(3, 5)),
                                           (2000, 1, 1, 40, 24, Fraction(1, 3))])
def test_extreme_shapes(T, E, k, h, I, rho):
    """A single token, a single expert, every token routed to every expert
    (k = E, up to the ABI's k = 32), the narrowest rows (h = I = 8) and
    rows that are no multiple of the 64-column swizzle atom."""
    inp = custom_inputs(T=T, E=E, k=k, h=h, I=I, s=0.5, rho=rho, seed=T + E + k)
    full_check(inp)
