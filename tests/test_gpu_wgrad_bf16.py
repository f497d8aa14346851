"""The weight gradient stored as bf16 (lrm_grouped_wgrad_bf16): the fp32
products in TMEM are those of lrm_grouped_wgrad, so every stored element is
that fp32 result rounded to nearest even, bit for bit; accumulate = 1 rounds
the fp32 sum with the stored values; experts with nothing retained get exact
zeros; and the result is within the path's relative Frobenius bound of the
oracle on the original inputs."""

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
from gpu_common import GEMM_RTOL, built_library, custom_inputs, need_gpu
from workloads import generate

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    built_library()


def _run(inp):
    from backward_token_expert_gb300.pipeline import Recalibration, to_device_inputs

    w = inp.workload
    rec = Recalibration(w.T, w.E, w.k, w.h, w.I, w.cf, w.rho)
    d = to_device_inputs(inp)
    rec.run(d["logits"], d["expert_idx"], d["g"], d["phi"], d["alpha"], d["W"])
    rec.wgrad_bf16()
    torch.cuda.synchronize()
    assert rec.device_status() == 0
    return rec


@pytest.mark.parametrize("case", ["tiny", "ragged", "qwen3"])
def test_bf16_dw_is_the_rounded_fp32_dw(case):
    if case == "tiny":
        inp = generate("tiny_T256_E8_k2_h64_I32")
    elif case == "ragged":
        inp = custom_inputs(T=3000, E=12, k=3, h=320, I=200, s=1.6, rho=Fraction(1, 2), seed=61, dead=2)
    else:
        inp = generate("qwen3_30b_a3b_T32768_E128_k8_h2048_I768")
    rec = _run(inp)
    try:
        expect = rec.buf.dW.to(torch.bfloat16)  # torch's fp32 -> bf16 is round to nearest even
        assert torch.equal(rec.dW_bf16.view(torch.int16), expect.view(torch.int16))
        so = rec.buf.sel_offsets.cpu().numpy()
        empty = np.flatnonzero(np.diff(so) == 0)
        for e in empty:
            assert torch.count_nonzero(rec.dW_bf16[int(e)]).item() == 0
        if case != "qwen3":
            w = inp.workload
            ids = rec.buf.sel_ids.cpu().numpy()[: so[-1]]
            ref = O.grouped_wgrad(inp.g, inp.phi, inp.alpha, so, ids, w.E, w.k)
            got = rec.dW_bf16.float().cpu().numpy()
            for e in range(w.E):
                if so[e + 1] > so[e]:
                    err = np.linalg.norm(got[e] - ref[e]) / np.linalg.norm(ref[e])
                    assert err <= GEMM_RTOL, (e, err)
    finally:
        rec.close()


def test_bf16_accumulate_rounds_the_fp32_sum():
    inp = custom_inputs(T=2000, E=10, k=2, h=128, I=96, seed=62)
    rec = _run(inp)
    try:
        gen = torch.Generator(device="cuda").manual_seed(5)
        start = torch.randn(rec.E, rec.h, rec.I, device="cuda", generator=gen).to(torch.bfloat16)
        rec.dW_bf16.copy_(start)
        rec.wgrad_bf16(accumulate=1)
        torch.cuda.synchronize()
        assert rec.device_status() == 0
        expect = (start.float() + rec.buf.dW).to(torch.bfloat16)
        assert torch.equal(rec.dW_bf16.view(torch.int16), expect.view(torch.int16))
    finally:
        rec.close()
