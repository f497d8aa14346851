"""Parity at the workloads' full sizes, in the launch configuration the bench
times.  Integer outputs are compared in full (counts, offsets, bucket, quotas,
selected ids); scores, compacted rows and GEMM outputs on seeded samples the
oracle computes one by one (sampled pairs, rows and experts, always including
the largest and the smallest non-empty expert and one whose row count is not
a multiple of the 128-row tile)."""

import numpy as np
import pytest

import oracle as O
from gpu_common import (
    GEMM_RTOL,
    SCORE_RTOL,
    built_library,
    check_compaction,
    check_gemms,
    check_route_stats,
    check_selection,
    need_gpu,
    rel_close,
    rel_fro,
    run_gpu,
)
from workloads import generate, get_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    built_library()


_SHARED = {}


def sweep_inputs(name):
    """The sweep points share one seed, so their g, phi and W are the same
    arrays: draw them once and only redo the routing of each point."""
    from workloads.generate import Inputs

    w = get_workload(name)
    if "base" not in _SHARED:
        _SHARED["base"] = generate(w)
    base = _SHARED["base"]
    r = generate(w, parts=())
    return Inputs(w, r.logits, r.expert_idx, r.alpha, base.g, base.phi, base.W, r.bias)


def check_padded(gpu, inp, so, ids, experts):
    """The zero-masked comparator (LRMoE sec. 3.4): every expert's slots hold
    its compacted rows then zeros (in full, bit for bit), the sampled experts'
    rows equal the oracle's compaction, and the GEMMs on the padded buffers
    match the oracle (sampled experts) and the compacted GEMMs (all experts)."""
    w = inp.workload
    C = gpu["C"]
    assert np.array_equal(gpu["pad_offsets"], np.arange(w.E + 1) * C)
    dpad = gpu["delta_pad"].reshape(w.E, C, w.h)
    ppad = gpu["phi_pad"].reshape(w.E, C, w.I)
    dphi_pad = gpu["dphi_pad"].reshape(w.E, C, w.I)
    for e in range(w.E):
        q = int(so[e + 1] - so[e])
        assert q <= C
        assert np.array_equal(dpad[e, :q], gpu["delta_c"][so[e]:so[e + 1]]), e
        assert np.array_equal(ppad[e, :q], gpu["phi_c"][so[e]:so[e + 1]]), e
        assert not dpad[e, q:].any() and not ppad[e, q:].any() and not dphi_pad[e, q:].any(), e
        ref = gpu["dW"][e].astype(np.float64)
        if q == 0:
            assert not gpu["dW_pad"][e].any()
        else:
            assert np.linalg.norm(gpu["dW_pad"][e] - ref) <= 1e-5 * np.linalg.norm(ref), e
    ref_dW = O.grouped_wgrad(inp.g, inp.phi, inp.alpha, so, ids, w.E, w.k, experts)
    ref_dphi = O.grouped_dgrad(inp.g, inp.W, inp.alpha, so, ids, w.E, w.k, experts)
    for e in experts:
        q = int(so[e + 1] - so[e])
        if q == 0:
            continue
        dc, pc, _ = O.compact(inp.g, inp.phi, inp.alpha, ids[so[e]:so[e + 1]], w.k)
        assert np.array_equal(dpad[e, :q], dc) and np.array_equal(ppad[e, :q], pc), e
        assert rel_fro(gpu["dW_pad"][e], ref_dW[e]) <= GEMM_RTOL, e
        assert rel_fro(O.bf16_to_f64(dphi_pad[e, :q]), ref_dphi[e]) <= GEMM_RTOL, e


def sampled_check(name, n_pairs=20000, n_rows=4096, n_random_experts=3, inp=None, padded=False):
    inp = generate(name) if inp is None else inp
    w = inp.workload
    gpu = run_gpu(inp, padded=padded)
    st = O.route_stats(inp.logits, inp.expert_idx, w.E, w.cf, w.rho)
    check_route_stats(gpu, inp, st)
    assert np.array_equal(gpu["quota"], st["quota"])
    rng = np.random.default_rng(1234)
    # scores on sampled pairs (the oracle evaluated pair by pair)
    u = np.sort(rng.choice(w.N, size=min(n_pairs, w.N), replace=False))
    R = O.score(inp.g[u // w.k], inp.phi[u], inp.alpha[u], 1)
    assert np.all(rel_close(gpu["score"][u], R, SCORE_RTOL, 1e-30))
    # selection in full, rerun on the GPU's fp32 scores
    so, ids = check_selection(gpu, inp, st["quota"])
    # compaction on sampled rows
    rows = np.sort(rng.choice(ids.size, size=min(n_rows, ids.size), replace=False))
    check_compaction(gpu, inp, ids, rows)
    # GEMMs on sampled experts
    q = np.diff(so)
    nz = np.flatnonzero(q > 0)
    experts = {int(nz[np.argmax(q[nz])]), int(nz[np.argmin(q[nz])])}
    ragged = nz[q[nz] % 128 != 0]
    if ragged.size:
        experts.add(int(ragged[0]))
    experts.update(int(e) for e in rng.choice(nz, size=min(n_random_experts, nz.size), replace=False))
    experts.update(int(e) for e in np.flatnonzero(q == 0))  # exact zeros
    worst = check_gemms(gpu, inp, so, ids, sorted(experts))
    if padded:
        check_padded(gpu, inp, so, ids, sorted(experts))
    return inp, gpu, st, worst


def test_qwen3_30b_a3b_layer():
    inp, gpu, st, worst = sampled_check("qwen3_30b_a3b_T32768_E128_k8_h2048_I768")
    # informational: selection on the fp64 scores differs from the parity-mode
    # selection only at near-ties of each expert's boundary score
    w = inp.workload
    R64 = O.score(inp.g, inp.phi, inp.alpha, w.k)
    so64, ids64 = O.select(R64, inp.expert_idx, w.E, st["quota"])
    e_u = inp.expert_idx.reshape(-1)
    for e in range(w.E):
        a = ids64[so64[e]:so64[e + 1]]
        b = gpu["sel_ids"][gpu["sel_offsets"][e]:gpu["sel_offsets"][e + 1]]
        diff = np.setxor1d(a, b)
        if diff.size:
            tau = R64[a].min()
            assert np.all(e_u[diff] == e)
            assert np.all(np.abs(R64[diff] - tau) <= 2e-5 * tau), e


def test_glm45_air_layer():
    sampled_check("glm45_air_T32768_E128_k8_h4096_I1408")


SWEEP = [f"qwen3_sweep_s{s:g}_rho{r}" for s in (0.0, 0.8, 1.2, 1.6) for r in ("1_1", "3_4", "1_2")]


@pytest.mark.parametrize("name", SWEEP)
def test_skew_sweep_point_with_zero_masked_comparator(name):
    # every point of the skew / retention sweep (Zipf s x rho on the
    # Qwen3-shaped layer): the compacted path and the capacity-padded
    # comparator that is timed against it on the same tensors
    inp, gpu, st, _ = sampled_check(name, n_random_experts=2, inp=sweep_inputs(name), padded=True)
    assert gpu["summary"]["retained"] == st["retained"]


def test_large_batch_stress_with_empty_and_oversized_experts():
    inp, gpu, st, _ = sampled_check("stress_T131072_E128_k8_h4096_I1408", n_random_experts=2)
    assert (st["counts"] == 0).sum() >= 1 and (st["counts"] > st["C"]).sum() >= 1


def test_deepseek_v2_layer():
    # E = 160 and k = 6: no power of two in the expert count, the pair count
    # per token or the per-block token count of route stats; h = 5120
    inp, gpu, st, _ = sampled_check("deepseek_v2_T32768_E160_k6_h5120_I1536")
    assert (st["counts"] > st["C"]).sum() >= 1


def test_gradient_l2_metric_at_full_size():
    # the ablation's gradient-only rule through the whole path of the bench workload
    from gpu_common import check_selection

    inp = generate("qwen3_30b_a3b_T32768_E128_k8_h2048_I768")
    w = inp.workload
    gpu = run_gpu(inp, metric=O.METRIC_GRAD_L2SQ)
    st = O.route_stats(inp.logits, inp.expert_idx, w.E, w.cf, w.rho)
    R = O.score_metric(O.METRIC_GRAD_L2SQ, inp.g, None, None, w.k, n_pairs=w.N)
    assert np.all(rel_close(gpu["score"], R, SCORE_RTOL, 1e-30))
    check_selection(gpu, inp, st["quota"])


def _qwen_inputs():
    if "qwen" not in _SHARED:
        _SHARED["qwen"] = generate("qwen3_30b_a3b_T32768_E128_k8_h2048_I768")
    return _SHARED["qwen"]


@pytest.mark.parametrize("pattern", ["all_but_one", "half", "one", "random"])
def test_selection_with_caller_quotas_at_full_size(pattern):
    """Per-expert selection of the bench layer under caller quotas that put
    each expert's boundary elsewhere than the rho rule does: near the lowest
    score (all but one kept, LRMoE Fig. 4's pattern), at the median (the
    boundary's top-11-bit bin then holds many keys), at the top (one kept) and
    at random ranks.  The ids must equal the oracle's selection on the GPU's
    fp32 scores in full, and the compacted rows its compaction on samples."""
    inp = _qwen_inputs()
    w = inp.workload
    n = np.bincount(inp.expert_idx.reshape(-1), minlength=w.E)
    rng = np.random.default_rng(99)
    quota = {"all_but_one": np.maximum(n - 1, 0), "half": (n + 1) // 2, "one": np.minimum(n, 1),
             "random": rng.integers(0, n + 1)}[pattern].astype(np.int32)
    gpu = run_gpu(inp, quota=quota)
    assert gpu["flags"] == 0
    assert np.array_equal(gpu["quota"], quota)
    so, ids = check_selection(gpu, inp, quota)
    assert gpu["sel_offsets"][-1] == quota.sum()
    rows = np.sort(rng.choice(ids.size, size=min(4096, ids.size), replace=False))
    check_compaction(gpu, inp, ids, rows)


def test_run_to_run_bit_identity_at_full_size():
    """Two runs of the bench layer give the same bits everywhere: no output
    depends on the order in which blocks or atomics happen to run."""
    inp = _qwen_inputs()
    a, b = run_gpu(inp), run_gpu(inp)
    assert a["flags"] == 0 and b["flags"] == 0
    for key in ("counts", "offsets", "bucket", "quota", "sel_offsets", "sel_ids", "delta_c", "phi_c", "dphi_c"):
        assert np.array_equal(a[key], b[key]), key
    for key in ("P", "f", "score", "alpha_c", "dW"):
        assert np.array_equal(a[key].view(np.uint32), b[key].view(np.uint32)), key
