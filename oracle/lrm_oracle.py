"""Plain fp64 CPU oracle of LRMoE's demand-side backward recalibration.

TEST INFRASTRUCTURE ONLY: the CUDA library never imports or calls this module;
tests, the smoke check and the bench's CPU-baseline leg do.  It shares no code,
constant or helper with the CUDA path; both read the same seeded inputs from
the ``workloads`` package, which holds none of the method's arithmetic.

Sources (cited by page title and the section / equation / figure):

* "LRMoE: Demand-Side Load Re-Calibration for Efficient MoE Training on
  Memory-Constrained Nodes" (Hu et al.), called LRMoE below:
  sec. 3.1 (quotas K_e with rho = sum K_e / N; compaction keeps the pairs in
  one fixed order and is described by per-expert counts and their prefix
  sums), sec. 3.2 Prop. 3.1 eq. (1)-(3) (the
  Load Recalibration Metric), sec. 3.3 Alg. 1 (score, per-expert
  TopK, compaction, packed expert backward), Fig. 4 and sec. 3.4 (variable-M
  grouped GEMMs without padding; equivalence with zero-masking), appendix 7.1
  eq. (4)-(12) (FC2 shapes, weighted cotangent delta_u = alpha_u g_t, rank-one
  factorisation), appendix 7.2 Prop. 7.1 (per-expert top-K is optimal, ties
  give several optimal sets), appendix 7.3 eq. (18)-(20).
* "Expert Parallel Math Deep" (aicassindra.com), called EPM below: sections
  "Routing as an expectation over a batch" (P_i, f_i), "Deriving the
  load-balancing auxiliary loss" (E * sum f_i P_i, range [1, E]) and
  "Capacity and the exact drop-rate formula" (C, drops, drop rate, E*C slots),
  with its worked example.

Readings where the pages leave a step open (each is also listed in the design
notes of the repository):

* quota rule: Q_e = ceil(rho * min(n_e, C)) with rho and CF exact rationals;
* capacity: C = floor(CF * N / E) in exact rational arithmetic;
* ties in the per-expert TopK go to the lower pair index u = t*k + j, and the
  retained ids of an expert are emitted in ascending u;
* the protected projection is FC2: W_e is [h, I], g_t is [h], phi_u is [I];
* compaction emits the weighted cotangent delta_u = bf16(fp32(alpha_u * g_t))
  (LRMoE eq. (5)), so neither GEMM applies alpha again;
* dW is kept in fp64 here (fp32 on the GPU), dphi likewise (bf16 on the GPU).

bf16 values are passed around as uint16 bit patterns.
"""

from __future__ import annotations

from fractions import Fraction

import numpy as np

__all__ = [
    "bf16_to_f64",
    "round_f64_to_bf16",
    "softmax_rows",
    "route_stats",
    "capacity_and_quotas",
    "aux_loss",
    "score",
    "score_metric",
    "random_scores",
    "splitmix64_outputs",
    "METRIC_LRM",
    "METRIC_GRAD_L2SQ",
    "METRIC_GRAD_L1",
    "METRIC_RANDOM",
    "select",
    "compact",
    "compact_padded",
    "grouped_wgrad",
    "grouped_dgrad",
    "grouped_wgrad_from_compact",
    "scatter_with_zeros",
    "silu",
    "swiglu_forward",
    "swiglu_backward",
    "fc1_backward",
    "combine_pairs",
    "grouped_dgrad_from_compact",
    "backward_recalibration",
]


# ---------------------------------------------------------------------------
# number formats


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (bf16 is the top half of an fp32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to fp32 (nearest-even), then to bf16 (nearest-even).

    This is the rounding the compaction step applies to alpha_u * g_t: the
    product is formed once in fp32 and then stored as bf16.  The second step
    adds half an ulp of bf16 (minus one, plus the kept lsb for the even case)
    to the fp32 bit pattern and truncates; NaN is outside the contract.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


# ---------------------------------------------------------------------------
# step 1: routing statistics and quotas (EPM; LRMoE sec. 3.1 / 3.3)


def softmax_rows(logits: np.ndarray) -> np.ndarray:
    """Gate probabilities p_i(x) = softmax(l)_i over all E experts (EPM)."""
    l = np.asarray(logits, dtype=np.float64)
    z = np.exp(l - l.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def aux_loss(f: np.ndarray, P: np.ndarray) -> float:
    """Unscaled load-balancing loss E * sum_i f_i P_i (EPM, auxiliary loss).

    The caller multiplies by its coefficient (about 0.01 on that page).
    """
    f = np.asarray(f, dtype=np.float64)
    P = np.asarray(P, dtype=np.float64)
    return float(f.size * np.sum(f * P))


def _ceil_div(a, b):
    return -((-a) // b)


def capacity_and_quotas(counts, N: int, E: int, cf=Fraction(5, 4), rho=Fraction(3, 4)):
    """C = floor(CF * N / E) in exact rationals (EPM, capacity section) and
    the quotas Q_e = ceil(rho * min(n_e, C)) of the routed counts n_e (LRMoE
    sec. 3.1 quotas, under the quota rule read above).  Returns (C, Q)."""
    cf = Fraction(cf)
    rho = Fraction(rho)
    C = (cf.numerator * N) // (cf.denominator * E)
    m = np.minimum(np.asarray(counts, dtype=np.int64), C)
    Q = _ceil_div(rho.numerator * m, rho.denominator).astype(np.int64)
    return C, Q


def route_stats(logits, expert_idx, E: int, cf=Fraction(5, 4), rho=Fraction(3, 4), quota=None):
    """Per-expert routing statistics, capacity, drop rate and retention quotas.

    * n_e = number of routed pairs on expert e (LRMoE Alg. 1);
    * P_e = mean over tokens of the full softmax, f_e = n_e / (T k), and
      aux = E * sum_e f_e P_e (EPM);
    * C = CF * T k / E (floor of the exact rational), dropped_e =
      max(0, n_e - C), drop rate = sum dropped / (T k), E*C padded slots and
      their utilisation (N - dropped) / (E C) (EPM, capacity section);
    * straggler factor n_max / mu with mu = T k / E (EPM);
    * quotas Q_e = ceil(rho * min(n_e, C)) unless ``quota`` is given, with
      realised rate sum Q / N (LRMoE sec. 3.1: rho = sum K_e / N);
    * a bucket of pair ids grouped by expert (ascending u inside an expert)
      and its prefix offsets: the per-expert counts and their prefix sums
      that LRMoE sec. 3.3 describes compaction with.
    """
    expert_idx = np.asarray(expert_idx)
    T, k = expert_idx.shape
    N = T * k
    e_u = expert_idx.reshape(-1).astype(np.int64)
    if e_u.size and (e_u.min() < 0 or e_u.max() >= E):
        raise ValueError("expert id out of range")
    if k > 1:
        srt = np.sort(expert_idx, axis=1)
        if np.any(srt[:, 1:] == srt[:, :-1]):
            raise ValueError("duplicate expert within a token")
    counts = np.bincount(e_u, minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    bucket = np.argsort(e_u, kind="stable").astype(np.int64)

    p = softmax_rows(logits)
    P = p.mean(axis=0)
    f = counts.astype(np.float64) / N
    aux = aux_loss(f, P)

    C, Q_rule = capacity_and_quotas(counts, N, E, cf, rho)
    over = np.maximum(counts - C, 0)
    dropped = int(over.sum())
    if quota is None:
        Q = Q_rule
    else:
        Q = np.asarray(quota, dtype=np.int64).copy()
        if Q.shape != (E,) or np.any(Q < 0) or np.any(Q > counts):
            raise ValueError("quota must satisfy 0 <= Q_e <= n_e")
    mu = Fraction(N, E)
    return dict(
        N=N,
        counts=counts,
        offsets=offsets,
        bucket=bucket,
        P=P,
        f=f,
        aux=aux,
        C=C,
        dropped=dropped,
        drop_rate=dropped / N,
        slots=E * C,
        util=(N - dropped) / (E * C) if C > 0 else 0.0,
        max_over_mean=float(Fraction(int(counts.max()), 1) / mu) if N else 0.0,
        quota=Q,
        retained=int(Q.sum()),
        rho_real=float(Q.sum()) / N if N else 0.0,
    )


# ---------------------------------------------------------------------------
# step 2: the Load Recalibration Metric (LRMoE sec. 3.2 eq. (3); app. 7.1 eq. (12))


def score(g_bits, phi_bits, alpha, k: int) -> np.ndarray:
    """R_u = alpha_u^2 * ||g_t||^2 * ||phi_u||^2 for every pair u = t*k + j.

    The squared Frobenius norm of the rank-one contribution
    G_u = (alpha_u g_t) phi_u^T factorises into the three squared norms
    (LRMoE eq. (11)), so no per-pair matrix is formed.  Computed in fp64 on
    the exact values of the bf16 / fp32 inputs.
    """
    g = bf16_to_f64(g_bits)
    phi = bf16_to_f64(phi_bits)
    a = np.asarray(alpha, dtype=np.float64)
    gn = np.einsum("ti,ti->t", g, g)
    pn = np.einsum("ui,ui->u", phi, phi)
    t_of_u = np.arange(a.size) // k
    return a * a * gn[t_of_u] * pn


# Selection metrics of LRMoE's ablation (sec. 4.7, Table 2).  The ablation
# compares the LRM with a squared L2 norm of the gradient, an absolute
# gradient magnitude and random drop; the gradient-only rules score a pair by
# its token's upstream gradient g_t alone (sec. 4.7: two pairs with the same
# upstream gradient norm get the same importance).  Readings: "|g|" is the L1
# sum sum_i |g_t,i|; random drop scores every pair with an independent
# uniform draw from the counter-based generator below.
METRIC_LRM, METRIC_GRAD_L2SQ, METRIC_GRAD_L1, METRIC_RANDOM = 0, 1, 2, 3

_M64 = (1 << 64) - 1
_GOLDEN = 0x9E3779B97F4A7C15


def splitmix64_outputs(state: int, count: int) -> list:
    """The first `count` outputs of the SplitMix64 generator from `state`
    (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
    OOPSLA 2014): add the golden-ratio increment to the state, then mix with
    two xor-shift-multiply steps and a final xor-shift."""
    out = []
    for _ in range(count):
        state = (state + _GOLDEN) & _M64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
        out.append(z ^ (z >> 31))
    return out


def random_scores(seed: int, n: int) -> np.ndarray:
    """Score of pair u: the (u+1)-th SplitMix64 output from state `seed`, top
    24 bits as a uniform value in [0, 1) (exact in fp32 and fp64)."""
    u = np.arange(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (np.uint64(seed & _M64) + (u + np.uint64(1)) * np.uint64(_GOLDEN))
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    return (z >> np.uint64(40)).astype(np.float64) * 2.0 ** -24


def score_metric(metric: int, g_bits, phi_bits, alpha, k: int, seed: int = 0, n_pairs=None) -> np.ndarray:
    """Per-pair selection score under one of the ablation's metrics."""
    if metric == METRIC_LRM:
        return score(g_bits, phi_bits, alpha, k)
    if metric == METRIC_RANDOM:
        n = int(n_pairs if n_pairs is not None else np.asarray(alpha).size)
        return random_scores(seed, n)
    g = bf16_to_f64(g_bits)
    per_token = np.einsum("ti,ti->t", g, g) if metric == METRIC_GRAD_L2SQ else np.abs(g).sum(axis=1)
    if metric not in (METRIC_GRAD_L2SQ, METRIC_GRAD_L1):
        raise ValueError(f"unknown metric {metric}")
    n = int(n_pairs if n_pairs is not None else g.shape[0] * k)
    return per_token[np.arange(n) // k]


# ---------------------------------------------------------------------------
# step 3: per-expert TopK within the quota (LRMoE sec. 3.2, Alg. 1, Prop. 7.1)


def select(R, expert_of_pair, E: int, quota):
    """Keep the Q_e highest-scoring pairs of every expert.

    Within expert e the candidates are all pairs routed to it; they are ranked
    by descending R and, among equal scores, by ascending pair index u.  The
    first Q_e are retained and emitted in ascending u ("consistent pair
    order").  Returns (sel_offsets[E+1], sel_ids[sum Q]).
    """
    R = np.asarray(R, dtype=np.float64)
    e_u = np.asarray(expert_of_pair).reshape(-1).astype(np.int64)
    Q = np.asarray(quota, dtype=np.int64)
    sel_offsets = np.concatenate([[0], np.cumsum(Q)]).astype(np.int64)
    sel_ids = np.empty(int(sel_offsets[-1]), dtype=np.int64)
    order_all = np.argsort(e_u, kind="stable")
    starts = np.concatenate([[0], np.cumsum(np.bincount(e_u, minlength=E))])
    for e in range(E):
        ids = order_all[starts[e]:starts[e + 1]]  # ascending u
        q = int(Q[e])
        if q > ids.size or q < 0:
            raise ValueError("quota must satisfy 0 <= Q_e <= n_e")
        rank = np.lexsort((ids, -R[ids]))  # primary: -R, secondary: u
        kept = np.sort(ids[rank[:q]])
        sel_ids[sel_offsets[e]:sel_offsets[e + 1]] = kept
    return sel_offsets, sel_ids


# ---------------------------------------------------------------------------
# step 4: physical compaction (LRMoE sec. 3.1 / 3.3 / 3.4, Fig. 4; eq. (5))


def compact(g_bits, phi_bits, alpha, sel_ids, k: int):
    """Gather retained rows into contiguous expert-major segments.

    Row r of the compacted buffers belongs to pair u = sel_ids[r], token
    t = u div k:  delta_c[r] = bf16(fp32(alpha_u * g_t)) (the weighted
    cotangent of LRMoE eq. (5)), phi_c[r] = phi_u (bit copy), alpha_c[r] =
    alpha_u.
    """
    ids = np.asarray(sel_ids, dtype=np.int64)
    a = np.asarray(alpha, dtype=np.float32)
    t = ids // k
    prod = a[ids].astype(np.float64)[:, None] * bf16_to_f64(np.asarray(g_bits)[t])
    delta_c = round_f64_to_bf16(prod)
    phi_c = np.asarray(phi_bits)[ids].copy()
    return delta_c, phi_c, a[ids].copy()


def compact_padded(delta_c, phi_c, sel_offsets, E: int, C: int):
    """Zero-masked fixed-shape layout of the same retained rows (LRMoE sec. 3.4).

    Expert e owns slots [e*C, (e+1)*C); its Q_e retained rows fill the first
    Q_e slots and the rest are zero.  Requires Q_e <= C.
    """
    so = np.asarray(sel_offsets, dtype=np.int64)
    h = delta_c.shape[1]
    I = phi_c.shape[1]
    dpad = np.zeros((E, C, h), dtype=np.uint16)
    ppad = np.zeros((E, C, I), dtype=np.uint16)
    for e in range(E):
        q = int(so[e + 1] - so[e])
        if q > C:
            raise ValueError("quota above capacity")
        dpad[e, :q] = delta_c[so[e]:so[e + 1]]
        ppad[e, :q] = phi_c[so[e]:so[e + 1]]
    return dpad, ppad


# ---------------------------------------------------------------------------
# step 5: packed expert backward of FC2 (LRMoE Alg. 1; app. 7.1 eq. (6)-(9))


def grouped_wgrad(g_bits, phi_bits, alpha, sel_offsets, sel_ids, E: int, k: int, experts=None):
    """dW_e = sum over retained u of (alpha_u g_t) phi_u^T, from the original inputs.

    Returns {e: [h, I] fp64}; experts with no retained pair give exact zeros.
    """
    so = np.asarray(sel_offsets, dtype=np.int64)
    ids_all = np.asarray(sel_ids, dtype=np.int64)
    a = np.asarray(alpha, dtype=np.float64)
    h = g_bits.shape[1]
    I = phi_bits.shape[1]
    out = {}
    for e in range(E) if experts is None else experts:
        ids = ids_all[so[e]:so[e + 1]]
        if ids.size == 0:
            out[e] = np.zeros((h, I))
            continue
        d = a[ids][:, None] * bf16_to_f64(g_bits[ids // k])
        out[e] = d.T @ bf16_to_f64(phi_bits[ids])
    return out


def grouped_dgrad(g_bits, W_bits, alpha, sel_offsets, sel_ids, E: int, k: int, experts=None):
    """dphi_u = alpha_u W_e^T g_t for every retained u of expert e (original inputs).

    Returns {e: [Q_e, I] fp64}, rows in the compacted (ascending u) order.
    """
    so = np.asarray(sel_offsets, dtype=np.int64)
    ids_all = np.asarray(sel_ids, dtype=np.int64)
    a = np.asarray(alpha, dtype=np.float64)
    out = {}
    for e in range(E) if experts is None else experts:
        ids = ids_all[so[e]:so[e + 1]]
        d = a[ids][:, None] * bf16_to_f64(g_bits[ids // k])
        out[e] = d @ bf16_to_f64(W_bits[e])
    return out


def scatter_with_zeros(rows, sel_ids, N: int) -> np.ndarray:
    """The inverse mapping of LRMoE (sec. 1 and 3.3; Alg. 1,
    ScatterWithZeros; sec. 3.4: kept rows return to their pairs' slots and
    dropped pairs' slots hold zeros for the next dense layer):
    row r of `rows` (the r-th retained pair in the compacted order) goes to
    row sel_ids[r] of an [N, width] array whose other rows are zero."""
    rows = np.asarray(rows)
    ids = np.asarray(sel_ids, dtype=np.int64)
    out = np.zeros((N,) + rows.shape[1:], dtype=rows.dtype)
    out[ids] = rows
    return out


# ---------------------------------------------------------------------------
# FC1 and its activation on the retained pairs (LRMoE sec. 3.4: the
# compacted row count sizes all four expert-backward GEMMs, the input- and
# weight-gradient products of FC1 and FC2).  The pages do not name the
# activation; it is read as SwiGLU: FC1 maps the expert input x_t to
# [a_u ; b_u] = W1_e x_t (W1_e is [2I, h], gate rows first), and the FC2
# input is phi_u = silu(a_u) * b_u with silu(a) = a / (1 + exp(-a)).


def silu(a):
    return a / (1.0 + np.exp(-a))


def swiglu_forward(ab):
    """phi = silu(a) * b for rows [a | b] of width 2I."""
    ab = np.asarray(ab, dtype=np.float64)
    I = ab.shape[1] // 2
    return silu(ab[:, :I]) * ab[:, I:]


def swiglu_backward(dphi, ab):
    """[da | db] for rows of phi = silu(a) * b: db = dphi * silu(a) and
    da = dphi * b * silu'(a), silu'(a) = s (1 + a (1 - s)), s = 1 / (1 + exp(-a))."""
    dphi = np.asarray(dphi, dtype=np.float64)
    ab = np.asarray(ab, dtype=np.float64)
    I = ab.shape[1] // 2
    a, b = ab[:, :I], ab[:, I:]
    sg = 1.0 / (1.0 + np.exp(-a))
    return np.concatenate([dphi * b * sg * (1.0 + a * (1.0 - sg)), dphi * a * sg], axis=1)


def fc1_backward(x, ab, W1, dphi_rows, sel_offsets, sel_ids, E: int, k: int, experts=None):
    """FC1 weight and input gradients of the retained pairs of every expert.

    x [T, h], ab [N, 2I] (the saved FC1 outputs [a | b] of every pair) and W1
    [E, 2I, h] are real arrays (convert bf16 bits with bf16_to_f64 first).
    dphi_rows[r] is the FC2 input gradient of the r-th retained pair (the
    compacted order).  For pair u = sel_ids[r] of expert e, token t = u div k:
    dh1_u = swiglu_backward(dphi_u, [a_u | b_u]); dW1_e = sum_u dh1_u x_t^T
    ([2I, h]); dx_u = W1_e^T dh1_u ([h]).  Returns ({e: dW1_e}, dx_rows) with
    dx_rows in the compacted order (rows of experts not in `experts` are 0).
    """
    so = np.asarray(sel_offsets, dtype=np.int64)
    ids_all = np.asarray(sel_ids, dtype=np.int64)
    x = np.asarray(x, dtype=np.float64)
    dh1 = swiglu_backward(dphi_rows, np.asarray(ab, dtype=np.float64)[ids_all])
    dW1 = {}
    dx = np.zeros((ids_all.size, x.shape[1]))
    for e in range(E) if experts is None else experts:
        r0, r1 = so[e], so[e + 1]
        dW1[e] = dh1[r0:r1].T @ x[ids_all[r0:r1] // k]
        dx[r0:r1] = dh1[r0:r1] @ np.asarray(W1[e], dtype=np.float64)
    return dW1, dx


def combine_pairs(rows, sel_ids, T: int, k: int) -> np.ndarray:
    """Input gradient of every token: the sum of the rows of its retained
    pairs (the inverse mapping followed by the MoE combine over the token's k
    experts); tokens without a retained pair get zeros."""
    rows = np.asarray(rows, dtype=np.float64)
    out = np.zeros((T, rows.shape[1]))
    np.add.at(out, np.asarray(sel_ids, dtype=np.int64) // k, rows)
    return out


def grouped_wgrad_from_compact(delta_c, phi_c, sel_offsets, E: int, experts=None):
    """dW_e = delta_c[seg e]^T phi_c[seg e] in fp64 on the compacted bf16 rows."""
    so = np.asarray(sel_offsets, dtype=np.int64)
    out = {}
    for e in range(E) if experts is None else experts:
        d = bf16_to_f64(delta_c[so[e]:so[e + 1]])
        p = bf16_to_f64(phi_c[so[e]:so[e + 1]])
        out[e] = d.T @ p
    return out


def grouped_dgrad_from_compact(delta_c, W_bits, sel_offsets, E: int, experts=None):
    """dphi_c[seg e] = delta_c[seg e] W_e in fp64 on the compacted bf16 rows."""
    so = np.asarray(sel_offsets, dtype=np.int64)
    out = {}
    for e in range(E) if experts is None else experts:
        d = bf16_to_f64(delta_c[so[e]:so[e + 1]])
        out[e] = d @ bf16_to_f64(W_bits[e])
    return out


# ---------------------------------------------------------------------------


def backward_recalibration(inputs, cf=None, rho=None, gemm_experts=None, R_for_selection=None):
    """Run the whole path in order: stats, score, select, compact, dgrad, wgrad.

    ``inputs`` is a ``workloads`` Inputs record.  ``R_for_selection`` replaces
    the fp64 scores in the selection step (used to rerun selection on another
    implementation's fp32 scores).  ``gemm_experts`` restricts the GEMMs to a
    subset of experts.
    """
    w = inputs.workload
    cf = w.cf if cf is None else cf
    rho = w.rho if rho is None else rho
    st = route_stats(inputs.logits, inputs.expert_idx, w.E, cf, rho)
    R = score(inputs.g, inputs.phi, inputs.alpha, w.k)
    Rs = R if R_for_selection is None else R_for_selection
    so, ids = select(Rs, inputs.expert_idx, w.E, st["quota"])
    dc, pc, ac = compact(inputs.g, inputs.phi, inputs.alpha, ids, w.k)
    dphi = grouped_dgrad(inputs.g, inputs.W, inputs.alpha, so, ids, w.E, w.k, gemm_experts)
    dW = grouped_wgrad(inputs.g, inputs.phi, inputs.alpha, so, ids, w.E, w.k, gemm_experts)
    return dict(stats=st, R=R, sel_offsets=so, sel_ids=ids, delta_c=dc, phi_c=pc, alpha_c=ac,
                dphi=dphi, dW=dW)
