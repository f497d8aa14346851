"""lrm_route_stats_noalloc: routing statistics for callers that cannot
allocate device memory.

Such a caller (for example one whose framework memory pool owns the whole GPU
and forbids outside allocations) can pass only its own inputs and outputs, so
this entry point keeps its scratch in a fixed array inside the library.  The
test calls it through the C ABI twice in a row, on two different layers, and
checks each result against lrm_route_stats with a caller workspace: integer
outputs bit for bit, fp32 outputs within the tolerance the parity tests use.
This file is collected last on purpose."""

from fractions import Fraction

import numpy as np
import pytest

from gpu_common import STAT_RTOL, built_library, custom_inputs, need_gpu, rel_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    built_library()


def _outputs(w, dev):
    import torch

    from backward_token_expert_gb300 import lrm as L

    i32 = dict(dtype=torch.int32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    return dict(counts=torch.full((w.E,), -7, **i32), offsets=torch.full((w.E + 1,), -7, **i32),
                bucket=torch.full((w.N,), -7, **i32), P=torch.full((w.E,), -1.0, **f32),
                f=torch.full((w.E,), -1.0, **f32), quota=torch.full((w.E,), -7, **i32),
                summary=torch.zeros(L.SUMMARY_BYTES, dtype=torch.uint8, device=dev))


def _compare(a, b):
    for key in ("counts", "offsets", "bucket", "quota", "summary"):
        assert np.array_equal(a[key].cpu().numpy(), b[key].cpu().numpy()), key
    for key in ("P", "f"):
        assert np.all(rel_close(a[key].cpu().numpy(), b[key].cpu().numpy(), STAT_RTOL, 1e-30)), key


def test_noalloc_route_stats_matches_workspace_version_twice():
    import torch

    from backward_token_expert_gb300 import lrm as L

    dev = "cuda:0"
    ctx = L.lrm_create(0)
    try:
        # calls in a row on one array: the second reuses what the first left, and
        # the third, a small layer with other E and k after the large one, reads
        # a scratch whose earlier contents span more blocks and another row pitch
        cases = [custom_inputs(T=3000, E=16, k=4, h=64, I=32, s=1.0, rho=Fraction(3, 4), seed=31),
                 custom_inputs(T=32768, E=128, k=8, h=64, I=32, s=0.8, rho=Fraction(3, 4), seed=32),
                 custom_inputs(T=700, E=24, k=3, h=64, I=32, s=1.2, rho=Fraction(1, 2), seed=33, dead=2)]
        for inp in cases:
            w = inp.workload
            dims = L.dims_of(w.T, w.E, w.k, w.h, w.I)
            logits = torch.from_numpy(inp.logits).to(dev)
            idx = torch.from_numpy(inp.expert_idx).to(dev)
            ref = _outputs(w, dev)
            ws_bytes = L.lrm_workspace_size(ctx, L.LRM_OP_ROUTE_STATS, dims)
            ws = torch.empty(max(256, ws_bytes), dtype=torch.uint8, device=dev)
            L.lrm_route_stats(ctx, logits, idx, dims, w.cf, w.rho, ref["counts"], ref["offsets"], ref["bucket"],
                              ref["P"], ref["f"], ref["quota"], ref["summary"], ws, ws.numel())
            got = _outputs(w, dev)
            L.lrm_route_stats_noalloc(ctx, logits, idx, dims, w.cf, w.rho, got["counts"], got["offsets"],
                                      got["bucket"], got["P"], got["f"], got["quota"], got["summary"])
            torch.cuda.synchronize()
            assert L.lrm_get_device_status(ctx) == 0
            _compare(got, ref)
        # a layer whose scratch would not fit is refused before any device work
        big = L.dims_of(1 << 22, 1024, 8, 64, 32)
        with pytest.raises(L.LrmError) as ei:
            L.lrm_route_stats_noalloc(ctx, 16, 16, big, Fraction(5, 4), Fraction(3, 4), 16, 16, 16, 16, 16, 16, 16)
        assert ei.value.code == L.LRM_ERR_SHAPE
    finally:
        L.lrm_destroy(ctx)
