"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and compare every step with the fp64 oracle on the same seeded inputs."""

from __future__ import annotations

import dataclasses
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
from workloads import generate, get_workload

torch = pytest.importorskip("torch")

SCORE_RTOL = 1e-5  # fp32 score vs fp64 (stated tolerance of the path)
STAT_RTOL = 1e-5  # importance / aux in fp32 vs fp64
GEMM_RTOL = 5e-3  # relative Frobenius error per expert, vs the oracle on the original inputs
WGRAD_TIGHT_RTOL = 1e-4  # fp32-accumulated dW vs fp64 on the same compacted bf16 rows


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    major, minor = torch.cuda.get_device_capability(0)
    if (major, minor) != (10, 3):
        pytest.skip(f"needs sm_103 (GB300), found sm_{major}{minor}")


def built_library():
    from backward_token_expert_gb300 import build

    build.build()


def bf16_np(t) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def workload(base="tiny_T256_E8_k2_h64_I32", **kw):
    return get_workload(base, **kw)


def run_gpu(inp, cf=None, rho=None, quota=None, max_rows=None, padded=False, metric=0, seed=0):
    """Run the whole path on cuda:0; returns numpy copies of every output."""
    from backward_token_expert_gb300 import lrm as L
    from backward_token_expert_gb300.pipeline import Recalibration, to_device_inputs

    w = inp.workload
    cf = Fraction(w.cf if cf is None else cf)
    rho = Fraction(w.rho if rho is None else rho)
    if quota is not None and max_rows is None:
        max_rows = w.N
    rec = Recalibration(w.T, w.E, w.k, w.h, w.I, cf, rho, max_rows=max_rows)
    try:
        d = to_device_inputs(inp)
        q = None if quota is None else torch.as_tensor(np.asarray(quota, dtype=np.int32), device="cuda")
        rec.route_stats(d["logits"], d["expert_idx"], quota_override=q)
        rec.backward_steps(d["g"], d["phi"], d["alpha"], d["W"], metric=metric, seed=seed)
        torch.cuda.synchronize()
        b = rec.buf
        so = b.sel_offsets.cpu().numpy().astype(np.int64)
        total = int(so[-1])
        out = dict(
            counts=b.counts.cpu().numpy(),
            offsets=b.offsets.cpu().numpy(),
            bucket=b.bucket.cpu().numpy()[: w.N],
            P=b.P.cpu().numpy(),
            f=b.f.cpu().numpy(),
            quota=b.quota.cpu().numpy(),
            summary=rec.summary(),
            score=b.score.cpu().numpy()[: w.N],
            sel_offsets=so,
            sel_ids=b.sel_ids.cpu().numpy()[:total].astype(np.int64),
            delta_c=bf16_np(b.delta_c[:total]),
            phi_c=bf16_np(b.phi_c[:total]),
            alpha_c=b.alpha_c[:total].cpu().numpy(),
            dphi_c=bf16_np(b.dphi_c[:total]),
            dW=b.dW.cpu().numpy(),
            max_rows=rec.max_rows,
            C=rec.C,
        )
        if padded:
            E, C = w.E, rec.C
            dpad = torch.empty(max(1, E * C), w.h, dtype=torch.bfloat16, device="cuda")
            ppad = torch.empty(max(1, E * C), w.I, dtype=torch.bfloat16, device="cuda")
            poff = torch.empty(E + 1, dtype=torch.int32, device="cuda")
            dphi_pad = torch.empty(max(1, E * C), w.I, dtype=torch.bfloat16, device="cuda")
            dW_pad = torch.empty(E, w.h, w.I, dtype=torch.float32, device="cuda")
            L.lrm_compact_padded(rec.ctx, b.delta_c, b.phi_c, b.sel_offsets, rec.dims, C, dpad, ppad, poff)
            L.lrm_grouped_dgrad(rec.ctx, dpad, d["W"], poff, rec.dims, E * C, dphi_pad)
            L.lrm_grouped_wgrad(rec.ctx, dpad, ppad, poff, rec.dims, E * C, 0, dW_pad)
            torch.cuda.synchronize()
            out.update(pad_offsets=poff.cpu().numpy(), delta_pad=bf16_np(dpad), phi_pad=bf16_np(ppad),
                       dphi_pad=bf16_np(dphi_pad), dW_pad=dW_pad.cpu().numpy())
        out["flags"] = rec.device_status()
        return out
    finally:
        rec.close()


def rel_close(a, ref, rtol, atol=0.0):
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return np.abs(a - ref) <= rtol * np.abs(ref) + atol


def rel_fro(x, ref) -> float:
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(np.asarray(x, np.float64) - ref) / n) if n > 0 else float(np.linalg.norm(x))


def check_route_stats(gpu, inp, st):
    assert gpu["flags"] == 0, gpu["flags"]
    assert np.array_equal(gpu["counts"], st["counts"])
    assert np.array_equal(gpu["offsets"], st["offsets"])
    assert np.array_equal(gpu["bucket"], st["bucket"])
    assert np.all(rel_close(gpu["P"], st["P"], STAT_RTOL, 1e-30))
    assert np.all(rel_close(gpu["f"], st["f"], 2.5e-7, 0))  # two fp32 roundings
    s = gpu["summary"]
    assert s["N"] == st["N"] and s["C"] == st["C"] and s["slots"] == st["slots"]
    assert s["dropped"] == st["dropped"]
    assert s["max_count"] == int(st["counts"].max()) and s["min_count"] == int(st["counts"].min())
    assert s["nonempty"] == int((st["counts"] > 0).sum())
    assert abs(s["aux_unscaled"] - st["aux"]) <= STAT_RTOL * st["aux"]
    assert abs(s["drop_rate"] - st["drop_rate"]) <= 2.5e-7 * max(st["drop_rate"], 1e-30) + 1e-12
    assert abs(s["util"] - st["util"]) <= 1e-6
    assert abs(s["max_over_mean"] - st["max_over_mean"]) <= 1e-6 * st["max_over_mean"]
    assert abs(s["sum_P"] - 1.0) <= 1e-5


def check_selection(gpu, inp, quota):
    w = inp.workload
    so, ids = O.select(gpu["score"].astype(np.float64), inp.expert_idx, w.E, quota)
    assert np.array_equal(gpu["sel_offsets"], so)
    assert np.array_equal(gpu["sel_ids"], ids)
    return so, ids


def check_compaction(gpu, inp, ids, rows=None):
    w = inp.workload
    rows = np.arange(ids.size) if rows is None else rows
    dc, pc, ac = O.compact(inp.g, inp.phi, inp.alpha, ids[rows], w.k)
    assert np.array_equal(gpu["delta_c"][rows], dc)
    assert np.array_equal(gpu["phi_c"][rows], pc)
    assert np.array_equal(gpu["alpha_c"][rows].view(np.uint32), ac.view(np.uint32))


def check_gemms(gpu, inp, so, ids, experts=None, dW_key="dW", dphi_key="dphi_c", dphi_offsets=None):
    w = inp.workload
    experts = range(w.E) if experts is None else experts
    ref_dW = O.grouped_wgrad(inp.g, inp.phi, inp.alpha, so, ids, w.E, w.k, experts)
    ref_dphi = O.grouped_dgrad(inp.g, inp.W, inp.alpha, so, ids, w.E, w.k, experts)
    tight = O.grouped_wgrad_from_compact(gpu["delta_c"], gpu["phi_c"], so, w.E, experts)
    poff = so if dphi_offsets is None else dphi_offsets
    worst = 0.0
    for e in experts:
        q = int(so[e + 1] - so[e])
        dW = gpu[dW_key][e]
        if q == 0:
            assert np.all(dW == 0), f"expert {e} has no retained row but a non-zero dW"
            continue
        err = rel_fro(dW, ref_dW[e])
        assert err <= GEMM_RTOL, (e, err)
        assert rel_fro(dW, tight[e]) <= WGRAD_TIGHT_RTOL, e
        dphi = O.bf16_to_f64(gpu[dphi_key][poff[e]:poff[e] + q])
        err2 = rel_fro(dphi, ref_dphi[e])
        assert err2 <= GEMM_RTOL, (e, err2)
        worst = max(worst, err, err2)
    return worst


def custom_inputs(T, E, k, h, I, s=1.0, rho=Fraction(3, 4), seed=0, phi_scale="uniform", dead=0):
    w = dataclasses.replace(get_workload("tiny_T256_E8_k2_h64_I32"), name=f"custom_T{T}_E{E}_k{k}_h{h}_I{I}", T=T,
                            E=E, k=k, h=h, I=I, zipf_s=s, rho=Fraction(rho), seed=seed, phi_scale=phi_scale,
                            dead_experts=dead)
    return generate(w)
