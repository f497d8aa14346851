"""Parity of the ablation's selection metrics (LRMoE sec. 4.7, Table 2) with
the oracle: the gradient-only scores within the score tolerance, the seeded
random scores bit for bit (both sides implement SplitMix64 from its
definition), and the rest of the path (selection, compaction, GEMMs) on the
GPU's scores exactly as for the LRM."""

from fractions import Fraction

import numpy as np
import pytest

import oracle as O
from gpu_common import (
    SCORE_RTOL,
    built_library,
    check_compaction,
    check_gemms,
    check_selection,
    custom_inputs,
    need_gpu,
    rel_close,
    run_gpu,
)

pytestmark = pytest.mark.gpu

METRICS = [O.METRIC_GRAD_L2SQ, O.METRIC_GRAD_L1, O.METRIC_RANDOM]


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    built_library()


def _check_metric(inp, metric, seed):
    w = inp.workload
    gpu = run_gpu(inp, metric=metric, seed=seed)
    assert gpu["flags"] == 0
    R = O.score_metric(metric, inp.g, inp.phi, inp.alpha, w.k, seed=seed, n_pairs=w.N)
    if metric == O.METRIC_RANDOM:
        assert np.array_equal(gpu["score"].astype(np.float64), R)
    else:
        assert np.all(rel_close(gpu["score"], R, SCORE_RTOL, 1e-30))
    st = O.route_stats(inp.logits, inp.expert_idx, w.E, w.cf, w.rho)
    so, ids = check_selection(gpu, inp, st["quota"])
    check_compaction(gpu, inp, ids)
    check_gemms(gpu, inp, so, ids)
    return gpu


@pytest.mark.parametrize("metric", METRICS)
def test_metric_ragged_tiles(metric):
    inp = custom_inputs(T=1536, E=16, k=4, h=320, I=200, s=1.0, rho=Fraction(3, 4), seed=21)
    _check_metric(inp, metric, seed=0xC0FFEE)


@pytest.mark.parametrize("metric", METRICS)
def test_metric_large_expert_sampled_bracket(metric):
    inp = custom_inputs(T=20000, E=2, k=1, h=64, I=32, s=0.0, rho=Fraction(3, 4), seed=22)
    _check_metric(inp, metric, seed=7)


def test_random_metric_seed_changes_the_draw():
    inp = custom_inputs(T=512, E=4, k=2, h=64, I=32, seed=23)
    a = run_gpu(inp, metric=O.METRIC_RANDOM, seed=1)["score"]
    b = run_gpu(inp, metric=O.METRIC_RANDOM, seed=2)["score"]
    assert not np.array_equal(a, b)
    assert np.array_equal(a.astype(np.float64), O.random_scores(1, a.size))
