"""The FC1 side of the expert backward on the retained pairs (LRMoE sec. 3.4;
SwiGLU read) against the oracle, run from the GPU's compacted FC2 input
gradient: dh1 elementwise within bf16 rounding, the FC1 input gradient of the
retained rows and the FC1 weight gradient per expert within the path's
relative Frobenius bound, and the token input gradient (the combine over each
token's retained pairs) likewise, with exact zeros for tokens that kept none."""

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
from gpu_common import bf16_np, built_library, custom_inputs, need_gpu
from workloads import fc1_inputs, generate

pytestmark = pytest.mark.gpu

FRO = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    built_library()


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _fc1_check(inp, f1, experts=None):
    from backward_token_expert_gb300.pipeline import Recalibration, to_device_inputs

    w = inp.workload
    rec = Recalibration(w.T, w.E, w.k, w.h, w.I, w.cf, w.rho)
    try:
        d = to_device_inputs(inp)
        rec.run(d["logits"], d["expert_idx"], d["g"], d["phi"], d["alpha"], d["W"])
        rec.fc1_backward(_dev(f1.x), _dev(f1.ab), _dev(f1.W1))
        torch.cuda.synchronize()
        assert rec.device_status() == 0
        b, f = rec.buf, rec.fc1
        so = b.sel_offsets.cpu().numpy().astype(np.int64)
        ids = b.sel_ids.cpu().numpy()[: so[-1]].astype(np.int64)
        dphi_c = bf16_np(b.dphi_c[: so[-1]])
        dh1 = bf16_np(f.dh1[: so[-1]])
        dxc = bf16_np(f.dxc[: so[-1]])
        dW1 = f.dW1.cpu().numpy()
        dx = O.bf16_to_f64(bf16_np(f.dx)) if experts is None else None
    finally:
        rec.close()
    # only the rows and experts that are checked go to fp64 (the full-size
    # layer's [a | b] and W1 are 0.8 GB of bf16 each)
    chk = range(w.E) if experts is None else experts
    so_c = np.zeros(w.E + 1, dtype=np.int64)
    for e in range(w.E):
        so_c[e + 1] = so_c[e] + (so[e + 1] - so[e] if e in chk else 0)
    rows = np.concatenate([np.arange(so[e], so[e + 1]) for e in chk]) if so_c[-1] else np.zeros(0, np.int64)
    ids_c = ids[rows]
    dphi_c, dh1 = O.bf16_to_f64(dphi_c[rows]), O.bf16_to_f64(dh1[rows])
    dxc_bits, dxc = dxc, np.zeros((so[-1], w.h))
    dxc[rows] = O.bf16_to_f64(dxc_bits[rows])
    ab_c = O.bf16_to_f64(f1.ab[ids_c])
    ref_dh1 = O.swiglu_backward(dphi_c, ab_c)
    tol = 2.0 ** -8 * np.abs(ref_dh1) + 1e-6 * (np.abs(ref_dh1).max() if ref_dh1.size else 0.0)
    assert np.all(np.abs(dh1 - ref_dh1) <= tol)
    # the oracle on the checked rows: pair ids renumbered to row positions (k = 1)
    W1 = {e: O.bf16_to_f64(f1.W1[e]) for e in chk}
    ref_dW1, ref_rows = O.fc1_backward(O.bf16_to_f64(f1.x[ids_c // w.k]), ab_c, W1, dphi_c, so_c,
                                       np.arange(rows.size), w.E, 1, list(chk))
    ref_dx_rows = np.zeros((so[-1], w.h))
    ref_dx_rows[rows] = ref_rows
    for e in chk:
        r0, r1 = so[e], so[e + 1]
        if r1 == r0:
            assert np.all(dW1[e] == 0)
            continue
        assert np.linalg.norm(dW1[e] - ref_dW1[e]) <= FRO * np.linalg.norm(ref_dW1[e]), e
        assert np.linalg.norm(dxc[r0:r1] - ref_dx_rows[r0:r1]) <= FRO * np.linalg.norm(ref_dx_rows[r0:r1]), e
    if experts is None:
        # the combine alone: the GPU's own rows summed, then rounded to bf16 once
        own = O.combine_pairs(dxc, ids, w.T, w.k)
        assert np.all(np.abs(dx - own) <= 2.0 ** -8 * np.abs(own) + 1e-6 * np.abs(own).max())
        ref_dx = O.combine_pairs(ref_dx_rows, ids, w.T, w.k)
        assert np.linalg.norm(dx - ref_dx) <= FRO * np.linalg.norm(ref_dx)
        none_kept = np.ones(w.T, dtype=bool)
        none_kept[ids // w.k] = False
        assert np.all(dx[none_kept] == 0)
        return none_kept
    return None


def test_fc1_tiny_workload():
    inp = generate("tiny_T256_E8_k2_h64_I32")
    _fc1_check(inp, fc1_inputs(inp.workload))


def test_fc1_ragged_sizes_and_empty_experts():
    inp = custom_inputs(T=3000, E=12, k=3, h=192, I=200, s=1.6, rho=Fraction(1, 2), seed=51, dead=2)
    none_kept = _fc1_check(inp, fc1_inputs(inp.workload))
    assert none_kept.any()


def test_fc1_non_power_of_two_k_and_wide_tiles():
    inp = custom_inputs(T=999, E=20, k=6, h=136, I=520, s=1.2, rho=Fraction(3, 5), seed=52)
    _fc1_check(inp, fc1_inputs(inp.workload))


def test_fc1_qwen3_layer_sampled_experts():
    inp = generate("qwen3_30b_a3b_T32768_E128_k8_h2048_I768")
    w = inp.workload
    st = O.route_stats(inp.logits, inp.expert_idx, w.E, w.cf, w.rho)
    q = np.asarray(st["quota"])
    nz = np.flatnonzero(q > 0)
    experts = sorted({int(nz[np.argmax(q[nz])]), int(nz[np.argmin(q[nz])]), int(nz[len(nz) // 2])})
    _fc1_check(inp, fc1_inputs(w), experts)


def test_fc1_deepseek_v2_layer_sampled_experts():
    # 2I = 3072 and h = 5120: the FC1 GEMMs with K = 3072 and 20 output tiles of h
    inp = generate("deepseek_v2_T32768_E160_k6_h5120_I1536")
    w = inp.workload
    st = O.route_stats(inp.logits, inp.expert_idx, w.E, w.cf, w.rho)
    q = np.asarray(st["quota"])
    nz = np.flatnonzero(q > 0)
    experts = sorted({int(nz[np.argmax(q[nz])]), int(nz[np.argmin(q[nz])])})
    _fc1_check(inp, fc1_inputs(w), experts)


def test_fc1_single_expert_top1():
    inp = custom_inputs(T=700, E=1, k=1, h=64, I=40, rho=Fraction(2, 3), seed=53)
    _fc1_check(inp, fc1_inputs(inp.workload))


def test_fc1_nothing_retained_gives_exact_zeros():
    from backward_token_expert_gb300.pipeline import Recalibration, to_device_inputs

    inp = custom_inputs(T=400, E=6, k=2, h=64, I=48, seed=54)
    w = inp.workload
    f1 = fc1_inputs(w)
    rec = Recalibration(w.T, w.E, w.k, w.h, w.I, w.cf, w.rho)
    try:
        d = to_device_inputs(inp)
        rec.route_stats(d["logits"], d["expert_idx"], quota_override=torch.zeros(w.E, dtype=torch.int32, device="cuda"))
        rec.backward_steps(d["g"], d["phi"], d["alpha"], d["W"])
        f = rec._fc1_buffers()
        f.dx.fill_(1.0)  # must come back as zeros
        f.dW1.fill_(1.0)
        rec.fc1_backward(_dev(f1.x), _dev(f1.ab), _dev(f1.W1))
        torch.cuda.synchronize()
        assert rec.device_status() == 0
        assert int(rec.buf.sel_offsets[-1].item()) == 0
        assert torch.count_nonzero(rec.fc1.dW1).item() == 0
        assert torch.count_nonzero(rec.fc1.dx).item() == 0
    finally:
        rec.close()
