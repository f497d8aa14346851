"""Seeded synthetic workloads shaped like the layers the LRMoE paper trains.

Shapes follow the model table of "TopoEP" (Table 1: Qwen3-30B-A3B has 128
experts, top-8, hidden 2048, expert intermediate 768; GLM-4.5-Air has 128
experts, top-8, hidden 4096, intermediate 1408) and the LRMoE paper's setup
(sec. 4.1: sequence 8192 x micro-batch 4 = 32768 tokens per GPU).  Skewed
routing follows TopoEP sec. 6.4: random logits plus a fixed expert-specific
bias.  Here the bias is a log-Zipf prior, bias_e = -s * ln(pi(e) + 1) for a
seeded permutation pi, so s = 0 is uniform routing.

Everything is drawn from numpy's PCG64 with SeedSequence(seed).spawn(6) in
the fixed order [perm, logits, g, phi, phi-scale, W].  Large arrays are drawn
in fixed-size chunks, each from its own child SeedSequence, so the values do
not depend on how many threads fill them.

bf16 tensors are returned as uint16 bit patterns (row-major numpy arrays);
fp32 values are rounded to bf16 with round-to-nearest-even.
"""

from __future__ import annotations

import concurrent.futures as _fut
import dataclasses
import os
from fractions import Fraction

import numpy as np

_CHUNK = 1 << 23  # elements per independently seeded chunk


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic MoE layer backward (the FC2 / down projection)."""

    name: str
    T: int  # tokens
    E: int  # experts
    k: int  # experts per token (top-k)
    h: int  # model hidden size (FC2 output, rows of W_e)
    I: int  # expert intermediate size (FC2 input, columns of W_e)
    zipf_s: float  # log-Zipf router bias exponent
    rho: Fraction  # retention ratio of the quota rule
    cf: Fraction = Fraction(5, 4)  # capacity factor
    phi_scale: str = "uniform"  # per-row scale of phi: "uniform" U(0.5,2) or "lognormal" exp(N(0,1))
    dead_experts: int = 0  # experts given a -1e4 bias so that no token routes to them
    seed: int = 0
    note: str = ""

    @property
    def N(self) -> int:
        return self.T * self.k


def _wl(name, T, E, k, h, I, s, rho, **kw):
    return Workload(name=name, T=T, E=E, k=k, h=h, I=I, zipf_s=s, rho=Fraction(rho), **kw)


WORKLOADS: dict[str, Workload] = {}


def _add(w: Workload) -> None:
    WORKLOADS[w.name] = w


_add(_wl("tiny_T256_E8_k2_h64_I32", 256, 8, 2, 64, 32, 1.0, Fraction(3, 4),
         note="small case the oracle finishes in seconds"))
_add(_wl("qwen3_30b_a3b_T32768_E128_k8_h2048_I768", 32768, 128, 8, 2048, 768, 0.8, Fraction(3, 4),
         note="Qwen3-30B-A3B-shaped MoE layer, all 128 experts on one GPU"))
_add(_wl("glm45_air_T32768_E128_k8_h4096_I1408", 32768, 128, 8, 4096, 1408, 1.2, Fraction(3, 5),
         phi_scale="lognormal", note="GLM-4.5-Air-shaped layer, log-normal phi row scales"))
for _s in (0.0, 0.8, 1.2, 1.6):
    for _rho in (Fraction(1), Fraction(3, 4), Fraction(1, 2)):
        _add(_wl(f"qwen3_sweep_s{_s:g}_rho{_rho.numerator}_{_rho.denominator}", 32768, 128, 8, 2048, 768,
                 _s, _rho, note="skew/retention sweep on Qwen3-30B-A3B shapes"))
_add(_wl("stress_T131072_E128_k8_h4096_I1408", 131072, 128, 8, 4096, 1408, 1.2, Fraction(1, 2),
         dead_experts=2, note="large batch with empty and over-capacity experts"))
_add(_wl("deepseek_v2_T32768_E160_k6_h5120_I1536", 32768, 160, 6, 5120, 1536, 1.0, Fraction(3, 4),
         note="DeepSeek-V2-shaped layer: E = 160 and k = 6 are not powers of two, wider h"))


def get_workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    if overrides:
        if "rho" in overrides:
            overrides["rho"] = Fraction(overrides["rho"])
        w = dataclasses.replace(w, **overrides)
    return w


# ---------------------------------------------------------------------------
# bf16 bit conversions (input preparation only)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest-even) and return the uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    out = np.empty(b.shape, dtype=np.uint16)
    flat_b = b.reshape(-1)
    flat_o = out.reshape(-1)
    for s in range(0, flat_b.size, _CHUNK):
        c = flat_b[s:s + _CHUNK]
        r = (c + np.uint32(0x7FFF) + ((c >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
        flat_o[s:s + _CHUNK] = r.astype(np.uint16)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------------------


def _threads() -> int:
    try:
        return max(1, min(16, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return 1


def _fill_bf16(ss: np.random.SeedSequence, n: int, scale_fn=None) -> np.ndarray:
    """n standard-normal draws (fp32), optionally scaled per element, as bf16 bits."""
    out = np.empty(n, dtype=np.uint16)
    nchunks = (n + _CHUNK - 1) // _CHUNK
    seeds = ss.spawn(nchunks)

    def work(i):
        s = i * _CHUNK
        e = min(n, s + _CHUNK)
        v = np.random.Generator(np.random.PCG64(seeds[i])).standard_normal(e - s, dtype=np.float32)
        if scale_fn is not None:
            v = scale_fn(v, s, e)
        out[s:e] = f32_to_bf16_bits(v)

    if nchunks == 1:
        work(0)
    else:
        with _fut.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nchunks)))
    return out


@dataclasses.dataclass
class Inputs:
    workload: Workload
    logits: np.ndarray  # [T, E] float32 router logits
    expert_idx: np.ndarray  # [T, k] int32, slot j = j-th highest logit
    alpha: np.ndarray  # [T*k] float32 gate weight of pair u = t*k + j
    g: np.ndarray | None  # [T, h] bf16 bits: gradient at the expert output, before alpha
    phi: np.ndarray | None  # [T*k, I] bf16 bits: saved input of FC2 for pair u
    W: np.ndarray | None  # [E, h, I] bf16 bits: FC2 weight W_e in R^{h x I}
    bias: np.ndarray  # [E] float64 router bias used


def routing(w: Workload):
    """Router logits, top-k expert ids and renormalised top-k gate weights."""
    ss = np.random.SeedSequence(w.seed).spawn(6)
    rng_perm = np.random.Generator(np.random.PCG64(ss[0]))
    perm = rng_perm.permutation(w.E)
    bias = -w.zipf_s * np.log(perm.astype(np.float64) + 1.0)
    if w.dead_experts:
        dead = rng_perm.choice(w.E, size=w.dead_experts, replace=False)
        bias[dead] = -1.0e4
    rng_l = np.random.Generator(np.random.PCG64(ss[1]))
    logits = (rng_l.standard_normal((w.T, w.E)) + bias[None, :]).astype(np.float32)
    # top-k by logit, ties to the lower expert id (stable sort of the negated logits)
    order = np.argsort(-logits, axis=1, kind="stable")[:, : w.k]
    expert_idx = order.astype(np.int32)
    sel = np.take_along_axis(logits, order, axis=1).astype(np.float64)
    z = np.exp(sel - sel.max(axis=1, keepdims=True))
    alpha = (z / z.sum(axis=1, keepdims=True)).astype(np.float32).reshape(-1)
    return logits, expert_idx, alpha, bias, ss


def generate(w: Workload | str, parts=("g", "phi", "W")) -> Inputs:
    if isinstance(w, str):
        w = get_workload(w)
    logits, expert_idx, alpha, bias, ss = routing(w)
    g = phi = W = None
    if "g" in parts:
        g = _fill_bf16(ss[2], w.T * w.h).reshape(w.T, w.h)
    if "phi" in parts:
        rng_sc = np.random.Generator(np.random.PCG64(ss[4]))
        if w.phi_scale == "uniform":
            row_scale = rng_sc.uniform(0.5, 2.0, size=w.N).astype(np.float32)
        elif w.phi_scale == "lognormal":
            row_scale = np.exp(rng_sc.standard_normal(w.N)).astype(np.float32)
        else:
            raise ValueError(w.phi_scale)
        I = w.I

        def scale_fn(v, s, e, row_scale=row_scale, I=I):
            rows = np.arange(s, e, dtype=np.int64) // I
            return v * row_scale[rows]

        phi = _fill_bf16(ss[3], w.N * w.I, scale_fn).reshape(w.N, w.I)
    if "W" in parts:
        W = _fill_bf16(ss[5], w.E * w.h * w.I,
                       lambda v, s, e: v * np.float32(0.02)).reshape(w.E, w.h, w.I)
    return Inputs(w, logits, expert_idx, alpha, g, phi, W, bias)


@dataclasses.dataclass
class Fc1Inputs:
    """The saved state of the FC1 side of the expert backward (SwiGLU read):
    the expert input of every token, the saved FC1 output [a | b] (gate, up)
    of every pair, and the FC1 weights.  They are drawn independently of the
    FC2 tensors of ``generate`` (the backward takes them as given)."""

    x: np.ndarray  # [T, h] bf16 bits: expert input of token t
    ab: np.ndarray  # [T*k, 2I] bf16 bits: saved FC1 output [a | b] of pair u
    W1: np.ndarray  # [E, 2I, h] bf16 bits: FC1 weight (gate rows first)


def fc1_inputs(w: Workload | str) -> Fc1Inputs:
    """x ~ N(0, 1), [a | b] ~ N(0, 1), W1 ~ N(0, 0.02^2), bf16; from the child
    seeds 6, 7, 8 of the workload's SeedSequence (children 0-5 feed
    ``generate``, so its tensors do not change)."""
    if isinstance(w, str):
        w = get_workload(w)
    ss = np.random.SeedSequence(w.seed).spawn(9)
    x = _fill_bf16(ss[6], w.T * w.h).reshape(w.T, w.h)
    ab = _fill_bf16(ss[7], w.N * 2 * w.I).reshape(w.N, 2 * w.I)
    W1 = _fill_bf16(ss[8], w.E * 2 * w.I * w.h, lambda v, s, e: v * np.float32(0.02)).reshape(w.E, 2 * w.I, w.h)
    return Fc1Inputs(x, ab, W1)
