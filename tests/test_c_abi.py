"""A plain C program (tests/c/abi_caller.c) calling liblrm through include/lrm.h:
the header compiles as C11 and the program links on any machine; on a GB300
the program runs the whole path on cudaMalloc'd buffers, and its outputs
match the oracle like the Python-driven path's."""

import os
import shutil
import struct
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp_path):
    if shutil.which("gcc") is None or not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime_api.h")):
        pytest.skip("gcc or the CUDA headers are missing")
    from backward_token_expert_gb300 import build

    lib = build.build()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / "abi_caller")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-I" + os.path.join(ROOT, "include"),
           "-I" + os.path.join(CUDA, "include"), os.path.join(ROOT, "tests", "c", "abi_caller.c"), "-L" + libdir,
           "-llrm", "-L" + os.path.join(CUDA, "lib64"), "-lcudart", "-Wl,-rpath," + libdir,
           "-Wl,-rpath," + os.path.join(CUDA, "lib64"), "-o", exe]
    out = subprocess.run(cmd, capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    return exe


def test_c_caller_compiles_links_and_probes(tmp_path):
    exe = _build(tmp_path)
    out = subprocess.run([exe, "--probe"], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.startswith("abi 1 create LRM_")


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["tiny", "ragged"])
def test_c_caller_runs_the_path(tmp_path, case):
    from gpu_common import GEMM_RTOL, custom_inputs, need_gpu
    from workloads import generate

    need_gpu()
    exe = _build(tmp_path)
    inp = generate("tiny_T256_E8_k2_h64_I32") if case == "tiny" else custom_inputs(
        T=1500, E=12, k=3, h=320, I=200, s=1.6, rho=Fraction(1, 2), seed=81, dead=2)
    w = inp.workload
    from backward_token_expert_gb300.pipeline import max_retained_rows

    max_rows = max_retained_rows(w.T, w.E, w.k, w.cf, w.rho)
    fin, fout = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(fin, "wb") as f:
        f.write(struct.pack("<10i", w.T, w.E, w.k, w.h, w.I, w.cf.numerator, w.cf.denominator, w.rho.numerator,
                            w.rho.denominator, max_rows))
        for a, dt in ((inp.logits, np.float32), (inp.expert_idx, np.int32), (inp.alpha, np.float32),
                      (inp.g, np.uint16), (inp.phi, np.uint16), (inp.W, np.uint16)):
            f.write(np.ascontiguousarray(a, dtype=dt).tobytes())
    out = subprocess.run([exe, str(fin), str(fout)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    raw = fout.read_bytes()
    off = 0

    def take(n, dt):
        nonlocal off
        a = np.frombuffer(raw, dtype=dt, count=n, offset=off)
        off += a.nbytes
        return a

    flags = int(take(1, np.uint32)[0])
    score = take(w.N, np.float32)
    so = take(w.E + 1, np.int32).astype(np.int64)
    ids = take(max_rows, np.int32)[: so[-1]].astype(np.int64)
    dphi = take(max_rows * w.I, np.uint16).reshape(max_rows, w.I)
    dW = take(w.E * w.h * w.I, np.float32).reshape(w.E, w.h, w.I)
    assert flags == 0
    st = O.route_stats(inp.logits, inp.expert_idx, w.E, w.cf, w.rho)
    so_ref, ids_ref = O.select(score.astype(np.float64), inp.expert_idx, w.E, st["quota"])
    assert np.array_equal(so, so_ref) and np.array_equal(ids, ids_ref)
    ref_dW = O.grouped_wgrad(inp.g, inp.phi, inp.alpha, so, ids, w.E, w.k)
    ref_dphi = O.grouped_dgrad(inp.g, inp.W, inp.alpha, so, ids, w.E, w.k)
    for e in range(w.E):
        if so[e + 1] == so[e]:
            assert np.all(dW[e] == 0)
            continue
        assert np.linalg.norm(dW[e] - ref_dW[e]) <= GEMM_RTOL * np.linalg.norm(ref_dW[e])
        got = O.bf16_to_f64(dphi[so[e]:so[e + 1]])
        assert np.linalg.norm(got - ref_dphi[e]) <= GEMM_RTOL * np.linalg.norm(ref_dphi[e])
