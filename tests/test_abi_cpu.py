"""Host-side checks of the C ABI that need no GPU: the library builds for
sm_103a, loads, exports every entry point include/lrm.h declares, and rejects
bad arguments before touching the device."""

import ctypes
import os
import re
import subprocess
from fractions import Fraction

import numpy as np
import pytest

from backward_token_expert_gb300 import build as B
from backward_token_expert_gb300 import lrm as L
import oracle as O

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "lrm.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:LRM_API\s+)?(?:lrm_status|const char\s*\*|int32_t)\s+(lrm_\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 16
    assert set(names) == set(L.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s(lrm_\w+)", out))
    assert exported == set(names), exported ^ set(names)


def test_build_targets_sm103a_only():
    gencode = [B.ARCH[i + 1] for i, a in enumerate(B.ARCH) if a == "-gencode"]
    assert gencode == ["arch=compute_103a,code=sm_103a"]


def test_abi_version_and_status_strings(lib):
    assert L.lrm_abi_version() == 1
    for code, name in enumerate(L.STATUS_NAMES):
        assert L.lrm_status_string(code) == name
    assert L.lrm_status_string(99) == "LRM_ERR_UNKNOWN"


def test_struct_layouts_match_header(lib):
    assert ctypes.sizeof(L.Dims) == 20
    assert ctypes.sizeof(L.RouteSummary) == 8 * 4 + 6 * 4


def test_null_context_is_rejected_without_device_work(lib):
    d = L.dims_of(16, 4, 2, 64, 32)
    out = ctypes.c_size_t()
    assert lib.lrm_workspace_size(None, 0, d, ctypes.byref(out)) == L.LRM_ERR_INVALID_ARG
    assert lib.lrm_score(None, 16, 16, 16, d, 16, None) == L.LRM_ERR_INVALID_ARG
    assert lib.lrm_select(None, 16, 16, 16, 16, d, 4, 16, 16, None, 0, None) == L.LRM_ERR_INVALID_ARG
    assert lib.lrm_compact(None, 16, 16, 16, 16, 16, d, 4, 16, 16, None, None) == L.LRM_ERR_INVALID_ARG
    assert lib.lrm_grouped_dgrad(None, 16, 16, 16, d, 4, 16, None) == L.LRM_ERR_INVALID_ARG
    assert lib.lrm_grouped_wgrad(None, 16, 16, 16, d, 4, 0, 16, None) == L.LRM_ERR_INVALID_ARG
    assert lib.lrm_get_device_status(None, None, ctypes.byref(ctypes.c_uint32())) == L.LRM_ERR_INVALID_ARG
    assert lib.lrm_set_wait_budget(None, 5) == L.LRM_ERR_INVALID_ARG
    assert lib.lrm_selftest_wait_timeout(None, 5, None) == L.LRM_ERR_INVALID_ARG
    assert lib.lrm_destroy(None) == L.LRM_OK
    assert lib.lrm_create(0, None) == L.LRM_ERR_INVALID_ARG


def test_python_wrapper_raises_on_error(lib):
    with pytest.raises(L.LrmError) as ei:
        L.lrm_sm_count(None)
    assert ei.value.code == L.LRM_ERR_INVALID_ARG


def test_capacity_query_matches_the_oracle_on_the_worked_example(lib, golden):
    # "Expert Parallel Math Deep" worked example: 8 experts, T k = 131072 routed
    # pairs, CF = 1.25 -> C = 20480; the oracle's C is the pin
    ex = golden("expert_parallel_math_worked_example.json")
    loads = np.asarray(ex["loads"], dtype=np.int64)
    E, N = loads.size, int(loads.sum())
    cf = Fraction(*ex["CF"])
    T, k = N // 2, 2
    ids = np.repeat(np.arange(E), loads)
    idx = np.stack([ids[:T], ids[T:]], axis=1)
    st = O.route_stats(np.zeros((T, E)), idx, E, cf, Fraction(3, 4))
    dims = L.dims_of(T, E, k, 8, 8)
    assert L.lrm_capacity(dims, cf) == st["C"] == ex["C"]
    assert st["retained"] <= L.lrm_max_rows(dims, cf, Fraction(3, 4))
    assert L.lrm_capacity(L.dims_of(32768, 128, 8, 2048, 768), Fraction(5, 4)) == 2560


def test_row_bound_covers_every_routing_and_is_reached(lib):
    rng = np.random.default_rng(0)
    reached = 0
    for _ in range(300):
        E = int(rng.integers(1, 20))
        k = int(rng.integers(1, E + 1))
        T = int(rng.integers(1, 200))
        cf = Fraction(int(rng.integers(1, 9)), int(rng.integers(1, 5)))
        rho = Fraction(int(rng.integers(0, 5)), 4)
        p = rng.dirichlet(np.ones(E) * (0.3 if rng.random() < 0.7 else 50.0))
        idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)])
        st = O.route_stats(np.zeros((T, E)), idx, E, cf, rho)
        dims = L.dims_of(T, E, k, 8, 8)
        assert L.lrm_capacity(dims, cf) == st["C"]
        bound = L.lrm_max_rows(dims, cf, rho)
        assert st["retained"] <= bound
        reached += st["retained"] == bound
    assert reached > 0  # the bound is tight for some routings


def test_capacity_queries_reject_bad_arguments(lib):
    d = L.dims_of(16, 4, 2, 64, 32)
    out = ctypes.c_int32()
    assert lib.lrm_capacity(d, 5, 4, None) == L.LRM_ERR_INVALID_ARG
    assert lib.lrm_capacity(d, 0, 4, ctypes.byref(out)) == L.LRM_ERR_INVALID_ARG
    assert lib.lrm_max_rows(d, 5, 4, 5, 4, ctypes.byref(out)) == L.LRM_ERR_INVALID_ARG  # rho > 1
    assert lib.lrm_max_rows(L.dims_of(16, 4, 2, 60, 32), 5, 4, 3, 4, ctypes.byref(out)) == L.LRM_ERR_ALIGN
    # E * C beyond int32
    assert lib.lrm_capacity(L.dims_of(1 << 20, 2, 2, 8, 8), 1 << 30, 1, ctypes.byref(out)) == L.LRM_ERR_SHAPE
