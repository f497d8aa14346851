"""HostPipeline (host buffers in, host buffers out, copies overlapping the
neighbouring batches' compute) gives, for every batch of a sequence, exactly
the results of the single-stream path on the same inputs, and on the small
layer the oracle's selection and GEMMs directly."""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_common import GEMM_RTOL, built_library, need_gpu, rel_fro
from workloads import generate, get_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    built_library()


def _host(inp):
    def t(a, dtype=None):
        x = torch.from_numpy(np.ascontiguousarray(a))
        return (x.view(dtype) if dtype is not None else x).pin_memory()

    return dict(logits=t(inp.logits), expert_idx=t(inp.expert_idx), alpha=t(inp.alpha),
                g=t(inp.g.view(np.int16), torch.bfloat16), phi=t(inp.phi.view(np.int16), torch.bfloat16),
                W=t(inp.W.view(np.int16), torch.bfloat16))


@pytest.mark.parametrize("name", ["tiny_T256_E8_k2_h64_I32", "qwen3_30b_a3b_T32768_E128_k8_h2048_I768"])
def test_every_batch_matches_the_single_stream_path(name):
    from backward_token_expert_gb300.pipeline import OUTPUT_NAMES, HostPipeline, Recalibration, to_device_inputs

    batches = [generate(get_workload(name, seed=s)) for s in (0, 1, 2)] if name.startswith("tiny") else \
        [generate(get_workload(name, seed=s)) for s in (0, 1)]
    w = batches[0].workload
    order = [0, 1, 2, 1, 0] if len(batches) == 3 else [0, 1, 0]
    pipe = HostPipeline(w.T, w.E, w.k, w.h, w.I, w.cf, w.rho)
    hin = [_host(b) for b in batches]
    outs = [pipe.host_outputs() for _ in order]
    try:
        for i, bi in enumerate(order):
            pipe.submit(hin[bi], outs[i])
        pipe.synchronize()
        assert pipe.device_status() == 0
    finally:
        pipe.close()
    rec = Recalibration(w.T, w.E, w.k, w.h, w.I, w.cf, w.rho)
    try:
        for bi, b in enumerate(batches):
            d = to_device_inputs(b)
            rec.run(d["logits"], d["expert_idx"], d["g"], d["phi"], d["alpha"], d["W"])
            torch.cuda.synchronize()
            rows = int(rec.buf.sel_offsets[-1].item())
            for i in (i for i, x in enumerate(order) if x == bi):
                o = outs[i]
                assert torch.equal(o["sel_offsets"], rec.buf.sel_offsets.cpu())
                assert torch.equal(o["sel_ids"][:rows], rec.buf.sel_ids[:rows].cpu())
                assert torch.equal(o["summary"], rec.buf.summary.cpu())
                assert torch.equal(o["dphi_c"][:rows].view(torch.int16), rec.buf.dphi_c[:rows].cpu().view(torch.int16))
                assert torch.equal(o["dW"], rec.buf.dW.cpu())
                if w.N <= 4096:
                    # and straight against the oracle: selection on this batch's fp32
                    # scores, then the GEMMs from the original inputs
                    st = O.route_stats(b.logits, b.expert_idx, w.E, w.cf, w.rho)
                    score = rec.buf.score[: w.N].cpu().numpy().astype(np.float64)
                    so, ids = O.select(score, b.expert_idx, w.E, st["quota"])
                    assert np.array_equal(o["sel_offsets"].numpy(), so)
                    assert np.array_equal(o["sel_ids"][:rows].numpy(), ids)
                    ref_dW = O.grouped_wgrad(b.g, b.phi, b.alpha, so, ids, w.E, w.k)
                    ref_dphi = O.grouped_dgrad(b.g, b.W, b.alpha, so, ids, w.E, w.k)
                    dphi = o["dphi_c"][:rows].float().numpy().astype(np.float64)
                    for e in range(w.E):
                        if so[e + 1] == so[e]:
                            assert not o["dW"][e].any()
                            continue
                        assert rel_fro(o["dW"][e].numpy(), ref_dW[e]) <= GEMM_RTOL, e
                        assert rel_fro(dphi[so[e]:so[e + 1]], ref_dphi[e]) <= GEMM_RTOL, e
        assert set(OUTPUT_NAMES) == set(outs[0])
    finally:
        rec.close()


@pytest.mark.parametrize("name", ["tiny_T256_E8_k2_h64_I32", "qwen3_30b_a3b_T32768_E128_k8_h2048_I768"])
def test_step_graph_replays_the_eager_step(name):
    # the graph is the launch configuration the bench times
    from backward_token_expert_gb300.pipeline import Recalibration, StepGraph, to_device_inputs

    a, b = (generate(get_workload(name, seed=s)) for s in (3, 4))
    w = a.workload
    rec = Recalibration(w.T, w.E, w.k, w.h, w.I, w.cf, w.rho)
    eager = Recalibration(w.T, w.E, w.k, w.h, w.I, w.cf, w.rho)
    try:
        d = to_device_inputs(a)
        graph = StepGraph(rec, d["logits"], d["expert_idx"], d["g"], d["phi"], d["alpha"], d["W"])
        for inp in (b, a, b):  # new batches written into the captured buffers
            src = to_device_inputs(inp)
            for name, t in graph.inputs.items():
                t.copy_(src[name])
            graph.replay()
            eager.run(src["logits"], src["expert_idx"], src["g"], src["phi"], src["alpha"], src["W"])
            torch.cuda.synchronize()
            assert torch.equal(rec.buf.sel_offsets, eager.buf.sel_offsets)
            rows = int(eager.buf.sel_offsets[-1].item())
            assert torch.equal(rec.buf.sel_ids[:rows], eager.buf.sel_ids[:rows])
            assert torch.equal(rec.buf.dW, eager.buf.dW)
            assert torch.equal(rec.buf.dphi_c[:rows].view(torch.int16), eager.buf.dphi_c[:rows].view(torch.int16))
        assert rec.device_status() == 0 and eager.device_status() == 0
    finally:
        rec.close()
        eager.close()
