"""Failure detection through the C ABI, with no GPU fault: bad data is flagged
in the device status word by the kernels' own checks, bad arguments are
rejected on the host, and a device wait that nothing completes gives up after
its time limit and reports LRM_ERR_TIMEOUT while the context stays usable."""

from fractions import Fraction

import numpy as np
import pytest

from gpu_common import built_library, check_gemms, check_selection, custom_inputs, need_gpu, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    built_library()


def _rec(T=64, E=4, k=2, h=64, I=32):
    from backward_token_expert_gb300.pipeline import Recalibration

    return Recalibration(T, E, k, h, I, Fraction(5, 4), Fraction(3, 4))


def test_bounded_wait_times_out_and_context_survives():
    import torch

    from backward_token_expert_gb300 import lrm as L

    rec = _rec()
    try:
        L.lrm_selftest_wait_timeout(rec.ctx, 2_000_000)  # 2 ms
        flags = rec.device_status()
        assert flags == (1 << L.LRM_ERR_TIMEOUT), L.flag_names(flags)
        assert rec.device_status() == 0  # reading clears the word
    finally:
        rec.close()
    # the device is still healthy: a normal run matches the oracle
    import oracle as O

    inp = custom_inputs(T=256, E=8, k=2, h=64, I=32, seed=20)
    gpu = run_gpu(inp)
    assert gpu["flags"] == 0
    st = O.route_stats(inp.logits, inp.expert_idx, 8, inp.workload.cf, inp.workload.rho)
    so, ids = check_selection(gpu, inp, st["quota"])
    check_gemms(gpu, inp, so, ids)
    assert torch.cuda.is_available()


def test_expert_id_out_of_range_is_flagged():
    import torch

    from backward_token_expert_gb300 import lrm as L

    rec = _rec()
    try:
        logits = torch.zeros(64, 4, device="cuda")
        idx = torch.tensor([[0, 1]] * 64, dtype=torch.int32, device="cuda")
        idx[5, 1] = 7  # outside [0, 4)
        rec.route_stats(logits, idx)
        flags = rec.device_status()
        assert flags & (1 << L.LRM_ERR_INDEX)
        assert rec.buf.counts.sum().item() == 127  # the bad pair is skipped
    finally:
        rec.close()


def test_duplicate_expert_within_token_is_flagged():
    import torch

    from backward_token_expert_gb300 import lrm as L

    rec = _rec()
    try:
        logits = torch.zeros(64, 4, device="cuda")
        idx = torch.tensor([[0, 1]] * 64, dtype=torch.int32, device="cuda")
        idx[9] = torch.tensor([2, 2], dtype=torch.int32)
        rec.route_stats(logits, idx)
        assert rec.device_status() & (1 << L.LRM_ERR_INDEX)
    finally:
        rec.close()


def test_quota_above_routed_count_is_clamped_and_flagged():
    import torch

    from backward_token_expert_gb300 import lrm as L

    inp = custom_inputs(T=256, E=8, k=2, h=64, I=32, seed=21)
    n = np.bincount(inp.expert_idx.reshape(-1), minlength=8)
    quota = n.copy()
    quota[3] = n[3] + 5
    gpu = run_gpu(inp, quota=quota)
    assert gpu["flags"] & (1 << L.LRM_ERR_QUOTA)
    assert gpu["sel_offsets"][4] - gpu["sel_offsets"][3] == n[3]
    assert torch.cuda.is_available()


def test_host_side_argument_errors():
    import torch

    from backward_token_expert_gb300 import lrm as L

    rec = _rec()
    try:
        g = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
        phi = torch.zeros(128, 32, dtype=torch.bfloat16, device="cuda")
        a = torch.zeros(128, device="cuda")
        with pytest.raises(L.LrmError) as ei:
            L.lrm_score(rec.ctx, g.data_ptr() + 2, phi, a, rec.dims, rec.buf.score)
        assert ei.value.code == L.LRM_ERR_ALIGN
        with pytest.raises(L.LrmError) as ei:
            L.lrm_route_stats(rec.ctx, torch.zeros(64, 4, device="cuda"), torch.zeros(64, 2, dtype=torch.int32,
                              device="cuda"), rec.dims, Fraction(5, 4), Fraction(3, 4), rec.buf.counts,
                              rec.buf.offsets, rec.buf.bucket, rec.buf.P, rec.buf.f, rec.buf.quota, rec.buf.summary,
                              rec.buf.ws_route, 8)
        assert ei.value.code == L.LRM_ERR_WORKSPACE
        with pytest.raises(L.LrmError) as ei:
            L.lrm_score(rec.ctx, g, phi, a, L.dims_of(64, 4, 2, 60, 32), rec.buf.score)
        assert ei.value.code == L.LRM_ERR_ALIGN
        with pytest.raises(L.LrmError) as ei:
            L.lrm_score(rec.ctx, g, phi, a, L.dims_of(64, 2000, 2, 64, 32), rec.buf.score)
        assert ei.value.code == L.LRM_ERR_SHAPE
        assert rec.device_status() == 0
    finally:
        rec.close()


def test_max_rows_too_small_is_flagged():
    from backward_token_expert_gb300 import lrm as L

    inp = custom_inputs(T=256, E=8, k=2, h=64, I=32, seed=22)
    gpu = run_gpu(inp, max_rows=16)
    assert gpu["flags"] & (1 << L.LRM_ERR_SHAPE)
