"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test ties one oracle function to something other than itself: a value
printed on a page (fixtures under tests/golden/, each with its source), a
closed form, an invariant, a special case that reduces to a different library
routine, or brute force on tiny inputs.
"""

import itertools
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
from workloads import f32_to_bf16_bits, generate, get_workload


def _worked_example_routing(ex):
    """Routing with the worked example's loads: sorted expert ids, token t takes
    positions t and t+T (distinct experts because every load is below T)."""
    T, k = ex["T"], ex["k"]
    ids = np.repeat(np.arange(ex["E"]), ex["loads"])
    assert ids.size == T * k
    return np.stack([ids[:T], ids[T:]], axis=1).astype(np.int32)


# ---------------------------------------------------------------------------
# selection metrics of the ablation (LRMoE sec. 4.7, Table 2)


def test_splitmix64_reference_sequence(golden):
    ref = golden("splitmix64_reference.json")
    got = O.splitmix64_outputs(ref["state"], len(ref["outputs_hex"]))
    assert got == [int(x, 16) for x in ref["outputs_hex"]]


def test_random_scores_are_the_generator_outputs_and_uniform():
    seed = 0x1234_5678_9ABC_DEF0
    n = 1 << 16
    r = O.random_scores(seed, n)
    # the vectorised draw equals the sequential generator (24 top bits of output u+1)
    seq = O.splitmix64_outputs(seed, 64)
    assert np.array_equal(r[:64], np.array([x >> 40 for x in seq], dtype=np.float64) * 2.0 ** -24)
    assert r.min() >= 0.0 and r.max() < 1.0
    # fp32 holds every value exactly
    assert np.array_equal(r.astype(np.float32).astype(np.float64), r)
    counts = np.bincount((r * 64).astype(np.int64), minlength=64)
    chi2 = ((counts - n / 64) ** 2 / (n / 64)).sum()
    assert chi2 < 120  # 63 degrees of freedom: far above the 99.99th percentile is a broken generator
    assert abs(np.corrcoef(r[:-1], r[1:])[0, 1]) < 0.02


def test_gradient_metrics_hand_values():
    g = f32_to_bf16_bits(np.array([[3.0, -4.0, 0.5, 0.0], [1.0, 1.0, 1.0, -1.0]], dtype=np.float32))
    l2 = O.score_metric(O.METRIC_GRAD_L2SQ, g, None, None, k=2, n_pairs=4)
    l1 = O.score_metric(O.METRIC_GRAD_L1, g, None, None, k=2, n_pairs=4)
    assert l2.tolist() == [25.25, 25.25, 4.0, 4.0]
    assert l1.tolist() == [7.5, 7.5, 4.0, 4.0]


def test_l2_metric_is_the_lrm_with_unit_alpha_and_phi():
    inp = generate("tiny_T256_E8_k2_h64_I32")
    w = inp.workload
    phi = np.zeros_like(inp.phi)
    phi[:, 3] = f32_to_bf16_bits(np.array([1.0], dtype=np.float32))[0]
    lrm = O.score(inp.g, phi, np.ones(w.N, dtype=np.float32), w.k)
    l2 = O.score_metric(O.METRIC_GRAD_L2SQ, inp.g, None, None, w.k, n_pairs=w.N)
    assert np.array_equal(lrm, l2)
    # and the L1 metric scales linearly and ignores signs
    g = inp.g.copy()
    l1 = O.score_metric(O.METRIC_GRAD_L1, g, None, None, w.k, n_pairs=w.N)
    g2 = g ^ np.uint16(0x8000)  # negate every bf16 value
    assert np.array_equal(O.score_metric(O.METRIC_GRAD_L1, g2, None, None, w.k, n_pairs=w.N), l1)
    g3 = f32_to_bf16_bits(2.0 * O.bf16_to_f64(g).astype(np.float32))
    assert np.array_equal(O.score_metric(O.METRIC_GRAD_L1, g3, None, None, w.k, n_pairs=w.N), 2.0 * l1)


# ---------------------------------------------------------------------------
# routing statistics: "Expert Parallel Math Deep", worked example and aux range


def test_worked_example_capacity_drops_utilisation(golden):
    ex = golden("expert_parallel_math_worked_example.json")
    idx = _worked_example_routing(ex)
    logits = np.zeros((ex["T"], ex["E"]), dtype=np.float32)
    st = O.route_stats(logits, idx, ex["E"], Fraction(*ex["CF"]), Fraction(3, 4))
    assert st["N"] == ex["total_dispatches"]
    assert st["N"] // ex["E"] == ex["mean_load"]
    assert st["counts"].tolist() == ex["loads"]
    assert st["C"] == ex["C"]
    assert st["dropped"] == ex["dropped"]
    assert round(100 * st["drop_rate"], 2) == ex["drop_rate_percent_rounded"]
    assert st["slots"] == ex["slots"]
    assert st["N"] - st["dropped"] == ex["real_carried"]
    assert round(100 * st["util"]) == ex["utilization_percent_rounded"]


def test_worked_example_aux_illustration(golden):
    """The page evaluates E * sum f_i P_i with P_i set equal to f_i and prints
    about 1.21 (sum f^2 printed as 0.1508, which is itself rounded/garbled:
    the loads give 0.15053).  Agreement to the page's ~1 % precision."""
    ex = golden("expert_parallel_math_worked_example.json")
    f = np.array(ex["loads"], dtype=np.float64) / ex["total_dispatches"]
    aux = O.aux_loss(f, f)
    assert abs(aux - ex["aux_illustration_rounded"]) <= 0.01
    assert abs(aux / ex["E"] - ex["aux_illustration_sum_f2_rounded"]) <= 5e-4


def test_worked_example_quotas_exact(golden):
    """Q_e = ceil(3/4 * min(n_e, C)) on the worked example, by hand:
    min(n, 20480) = [20480, 20480, 20000, 16000, 14000, 12000, 8000, 7072]."""
    ex = golden("expert_parallel_math_worked_example.json")
    idx = _worked_example_routing(ex)
    logits = np.zeros((ex["T"], ex["E"]), dtype=np.float32)
    st = O.route_stats(logits, idx, ex["E"], Fraction(5, 4), Fraction(3, 4))
    assert st["quota"].tolist() == [15360, 15360, 15000, 12000, 10500, 9000, 6000, 5304]
    assert st["retained"] == 88524
    # uniform logits: P_e = 1/E exactly, so aux = sum f = 1
    assert st["aux"] == pytest.approx(1.0, abs=1e-12)


def test_aux_is_one_at_uniform_load():
    """Balanced optimum of the aux loss is 1 (EPM, auxiliary loss section)."""
    T, k, E = 64, 4, 8
    idx = ((np.arange(T)[:, None] * k + np.arange(k)[None, :]) % E).astype(np.int32)
    logits = np.full((T, E), 0.25, dtype=np.float32)
    st = O.route_stats(logits, idx, E)
    assert np.all(st["counts"] == T * k // E)
    assert st["aux"] == pytest.approx(1.0, abs=1e-12)
    assert st["max_over_mean"] == 1.0


def test_aux_is_E_at_collapse():
    """Total collapse gives E (k = 1: every token on expert 0 with p_0 = 1)."""
    T, E = 32, 16
    idx = np.zeros((T, 1), dtype=np.int32)
    logits = np.full((T, E), -200.0, dtype=np.float32)
    logits[:, 0] = 0.0
    st = O.route_stats(logits, idx, E)
    assert st["aux"] == pytest.approx(E, rel=1e-12)
    assert st["max_over_mean"] == E


def test_importance_and_load_sum_to_one():
    rng = np.random.default_rng(1)
    T, E, k = 300, 12, 3
    logits = rng.standard_normal((T, E)).astype(np.float32) * 3
    idx = np.argsort(-logits, axis=1, kind="stable")[:, :k].astype(np.int32)
    st = O.route_stats(logits, idx, E)
    assert st["f"].sum() == pytest.approx(1.0, abs=1e-15)
    assert st["P"].sum() == pytest.approx(1.0, abs=1e-12)
    assert st["counts"].sum() == T * k
    # importance is the mean gate mass: compare with scipy's softmax
    sp = pytest.importorskip("scipy.special")
    assert np.allclose(st["P"], sp.softmax(logits.astype(np.float64), axis=1).mean(0), rtol=1e-13)


def test_quota_rule_uses_exact_rationals():
    """ceil(0.6 * 5) must be 3; a float product (3.0000000000000004) would give 4."""
    idx = np.array([[0], [0], [0], [0], [0], [1], [1], [1], [2], [3]], dtype=np.int32)
    st = O.route_stats(np.zeros((10, 4), np.float32), idx, 4, cf=Fraction(4), rho=Fraction(3, 5))
    assert st["counts"].tolist() == [5, 3, 1, 1]
    assert st["C"] == 10
    assert st["quota"].tolist() == [3, 2, 1, 1]


def test_quota_capped_by_capacity_and_bucket_is_stable():
    idx = np.array([[0, 1], [0, 2], [0, 1], [3, 0], [0, 2]], dtype=np.int32)
    st = O.route_stats(np.zeros((5, 4), np.float32), idx, 4, cf=Fraction(1), rho=Fraction(1))
    # C = 1 * 10 / 4 -> floor 2
    assert st["C"] == 2
    assert st["counts"].tolist() == [5, 2, 2, 1]
    assert st["dropped"] == 3
    assert st["quota"].tolist() == [2, 2, 2, 1]
    # bucket: expert-major, ascending pair index u = t*k + j
    assert st["bucket"].tolist() == [0, 2, 4, 7, 8, 1, 5, 3, 9, 6]
    assert st["offsets"].tolist() == [0, 5, 7, 9, 10]


def test_route_stats_rejects_bad_ids():
    with pytest.raises(ValueError):
        O.route_stats(np.zeros((2, 4), np.float32), np.array([[0, 4], [1, 2]], np.int32), 4)
    with pytest.raises(ValueError):
        O.route_stats(np.zeros((2, 4), np.float32), np.array([[1, 1], [1, 2]], np.int32), 4)


# ---------------------------------------------------------------------------
# score: Prop. 3.1 / eq. (11)-(12), by brute-force outer products


def _tiny(T=6, k=2, E=3, h=5, I=4, seed=3):
    rng = np.random.default_rng(seed)
    g = f32_to_bf16_bits(rng.standard_normal((T, h)).astype(np.float32))
    phi = f32_to_bf16_bits((rng.standard_normal((T * k, I)) * 1.5).astype(np.float32))
    W = f32_to_bf16_bits((rng.standard_normal((E, h, I)) * 0.1).astype(np.float32))
    alpha = rng.uniform(0.05, 1.0, T * k).astype(np.float32)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    return g, phi, W, alpha, idx


def test_score_equals_frobenius_norm_of_outer_product():
    g, phi, _, alpha, _ = _tiny(T=7, k=3, h=9, I=6)
    R = O.score(g, phi, alpha, 3)
    gf = O.bf16_to_f64(g)
    pf = O.bf16_to_f64(phi)
    for u in range(alpha.size):
        G = np.outer(float(alpha[u]) * gf[u // 3], pf[u])
        fro2 = sum(float(x) * float(x) for x in G.reshape(-1))
        assert R[u] == pytest.approx(fro2, rel=1e-12)


def test_score_zero_cases():
    g, phi, _, alpha, _ = _tiny()
    alpha = alpha.copy()
    alpha[0] = 0.0
    g = g.copy()
    g[1] = 0  # token 1: all-zero gradient -> both of its pairs score 0
    R = O.score(g, phi, alpha, 2)
    assert R[0] == 0.0 and R[2] == 0.0 and R[3] == 0.0
    assert np.all(R[4:] > 0)


# ---------------------------------------------------------------------------
# selection: Fig. 4, Prop. 7.1 (optimality, ties), invariants


def test_fig4_counts_offsets(golden):
    fx = golden("lrmoe_fig4_compaction.json")
    e_u = np.array(fx["pair_experts"], dtype=np.int32)
    idx = e_u.reshape(-1, 1)
    st = O.route_stats(np.zeros((e_u.size, 3), np.float32), idx, 3, quota=fx["retained_counts"])
    assert st["counts"].tolist() == fx["original_loads"]
    R = np.arange(e_u.size, 0, -1, dtype=np.float64)  # any scores
    so, ids = O.select(R, e_u, 3, st["quota"])
    assert so.tolist() == fx["offsets"]
    rows = np.diff(so).tolist()
    assert rows == [fx["segment_rows"]["e0"], fx["segment_rows"]["e1"], fx["segment_rows"]["e2"]]
    # every retained id belongs to its segment's expert, ascending inside a segment
    for e in range(3):
        seg = ids[so[e]:so[e + 1]]
        assert np.all(e_u[seg] == e) and np.all(np.diff(seg) > 0)


def test_select_maximises_retained_score_by_brute_force():
    """Prop. 7.1: any size-Q set of largest scores maximises the retained sum;
    with a strict boundary gap that set is unique and equals the oracle's."""
    rng = np.random.default_rng(7)
    for trial in range(40):
        n = int(rng.integers(1, 11))
        R = rng.choice([0.5, 1.0, 2.0, 3.0, 5.0, 8.0], size=n) if trial % 2 else rng.random(n)
        q = int(rng.integers(0, n + 1))
        e_u = np.zeros(n, dtype=np.int32)
        _, ids = O.select(R, e_u, 1, [q])
        best = max(sum(R[list(c)]) for c in itertools.combinations(range(n), q))
        assert sum(R[ids]) == pytest.approx(best, rel=1e-14, abs=0)
        srt = np.sort(R)[::-1]
        if 0 < q < n and srt[q - 1] > srt[q]:
            opt = [c for c in itertools.combinations(range(n), q) if sum(R[list(c)]) == best]
            assert len(opt) == 1 and list(opt[0]) == ids.tolist()


def test_select_ties_go_to_lower_pair_index():
    R = np.array([1.0, 2.0, 2.0, 2.0, 0.5, 2.0])
    e_u = np.zeros(6, dtype=np.int32)
    _, ids = O.select(R, e_u, 1, [2])
    assert ids.tolist() == [1, 2]
    _, ids = O.select(np.ones(6), e_u, 1, [4])
    assert ids.tolist() == [0, 1, 2, 3]


def test_select_invariants_per_expert():
    rng = np.random.default_rng(11)
    E, N = 5, 200
    e_u = rng.integers(0, E, N).astype(np.int32)
    R = np.round(rng.random(N) * 20) / 4  # many ties
    n = np.bincount(e_u, minlength=E)
    Q = np.array([rng.integers(0, c + 1) for c in n])
    so, ids = O.select(R, e_u, E, Q)
    assert np.all(np.diff(so) == Q)
    for e in range(E):
        kept = ids[so[e]:so[e + 1]]
        cand = np.flatnonzero(e_u == e)
        dropped = np.setdiff1d(cand, kept)
        assert np.all(e_u[kept] == e) and np.all(np.diff(kept) > 0)
        if kept.size and dropped.size:
            assert R[kept].min() >= R[dropped].max()
            tau = R[kept].min()
            # ties at the boundary: retained tied ids precede dropped tied ids
            if np.any(R[dropped] == tau):
                assert kept[R[kept] == tau].max() < dropped[R[dropped] == tau].min()


# ---------------------------------------------------------------------------
# compaction: rounding, bit copies, offsets


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    base = rng.standard_normal(4000).astype(np.float32).view(np.uint32)
    # force exact halfway cases with both parities of the kept lsb
    ties = (base & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    vals = np.concatenate([base, ties, np.array([0x00000001, 0x80000001, 0x7F7FFFFF], np.uint32)]).view(np.float32)
    mine = O.round_f64_to_bf16(vals.astype(np.float64))
    ref = torch.from_numpy(vals.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


def test_compaction_special_cases():
    g, phi, _, alpha, idx = _tiny(T=8, k=2, E=3)
    ids = np.array([5, 0, 9, 14, 3])
    # alpha = 1: the weighted cotangent is the gradient row itself
    dc, pc, ac = O.compact(g, phi, np.ones_like(alpha), ids, 2)
    assert np.array_equal(dc, g[ids // 2]) and np.array_equal(pc, phi[ids]) and np.all(ac == 1)
    # alpha = 1/2: exact halving, i.e. the bf16 exponent drops by one
    dc, _, _ = O.compact(g, phi, np.full_like(alpha, 0.5), ids, 2)
    src = g[ids // 2].astype(np.int32)
    expo = (src >> 7) & 0xFF
    ok = expo > 1
    assert np.array_equal(dc.astype(np.int32)[ok], (src - (1 << 7))[ok])


# ---------------------------------------------------------------------------
# grouped GEMMs: brute force, rank one, dense MoE special case, zero-masking, eq. (19)-(20)


def test_wgrad_dgrad_brute_force_loops():
    g, phi, W, alpha, idx = _tiny(T=5, k=2, E=3, h=4, I=3)
    e_u = idx.reshape(-1)
    Q = [min(2, int(c)) for c in np.bincount(e_u, minlength=3)]
    R = O.score(g, phi, alpha, 2)
    so, ids = O.select(R, e_u, 3, Q)
    dW = O.grouped_wgrad(g, phi, alpha, so, ids, 3, 2)
    dphi = O.grouped_dgrad(g, W, alpha, so, ids, 3, 2)
    gf, pf, Wf = O.bf16_to_f64(g), O.bf16_to_f64(phi), O.bf16_to_f64(W)
    for e in range(3):
        seg = ids[so[e]:so[e + 1]].tolist()
        for i in range(4):
            for j in range(3):
                acc = 0.0
                for u in seg:
                    acc += float(alpha[u]) * gf[u // 2, i] * pf[u, j]
                assert dW[e][i, j] == pytest.approx(acc, rel=1e-12, abs=1e-300)
        for r, u in enumerate(seg):
            for j in range(3):
                acc = sum(Wf[e, i, j] * float(alpha[u]) * gf[u // 2, i] for i in range(4))
                assert dphi[e][r, j] == pytest.approx(acc, rel=1e-12, abs=1e-300)


def test_single_pair_is_rank_one_outer_product():
    g, phi, W, alpha, idx = _tiny(T=4, k=2, E=4, h=6, I=5)
    e_u = idx.reshape(-1)
    counts = np.bincount(e_u, minlength=4)
    Q = (counts > 0).astype(np.int64)
    so, ids = O.select(O.score(g, phi, alpha, 2), e_u, 4, Q)
    dW = O.grouped_wgrad(g, phi, alpha, so, ids, 4, 2)
    for e in range(4):
        if Q[e]:
            u = int(ids[so[e]])
            ref = np.outer(float(alpha[u]) * O.bf16_to_f64(g[u // 2]), O.bf16_to_f64(phi[u]))
            assert np.allclose(dW[e], ref, rtol=1e-14, atol=0)
            assert np.linalg.matrix_rank(dW[e]) == 1
        else:
            assert np.all(dW[e] == 0)


def test_full_retention_equals_dense_moe_fc2_gradient():
    """rho = 1 with C >= max n_e keeps every pair: the result is the ordinary
    dense MoE FC2 backward, written here with a one-hot dispatch tensor."""
    T, k, E, h, I = 12, 2, 4, 6, 5
    g, phi, W, alpha, idx = _tiny(T=T, k=k, E=E, h=h, I=I, seed=9)
    logits = np.zeros((T, E), np.float32)
    st = O.route_stats(logits, idx, E, cf=Fraction(4), rho=Fraction(1))
    assert np.all(st["quota"] == st["counts"])
    so, ids = O.select(O.score(g, phi, alpha, k), idx, E, st["quota"])
    dW = O.grouped_wgrad(g, phi, alpha, so, ids, E, k)
    dphi = O.grouped_dgrad(g, W, alpha, so, ids, E, k)
    onehot = np.zeros((T * k, E))
    onehot[np.arange(T * k), idx.reshape(-1)] = 1.0
    gu = O.bf16_to_f64(g)[np.arange(T * k) // k]
    dense_dW = np.einsum("ue,u,ui,uj->eij", onehot, alpha.astype(np.float64), gu, O.bf16_to_f64(phi))
    dense_dphi = np.einsum("ue,u,ui,eij->uj", onehot, alpha.astype(np.float64), gu, O.bf16_to_f64(W))
    for e in range(E):
        assert np.allclose(dW[e], dense_dW[e], rtol=1e-12, atol=1e-14)
        seg = ids[so[e]:so[e + 1]]
        assert np.allclose(dphi[e], dense_dphi[seg], rtol=1e-12, atol=1e-14)


def test_scatter_with_zeros_is_the_dense_input_gradient_with_dropped_rows_zero():
    """The inverse mapping puts every retained row back at its pair: with full
    retention it equals the dense MoE FC2 input gradient written with a one-hot
    dispatch tensor; with a quota, the retained rows equal that dense gradient
    and every dropped row is zero."""
    T, k, E, h, I = 12, 2, 4, 6, 5
    g, phi, W, alpha, idx = _tiny(T=T, k=k, E=E, h=h, I=I, seed=9)
    N = T * k
    onehot = np.zeros((N, E))
    onehot[np.arange(N), idx.reshape(-1)] = 1.0
    gu = O.bf16_to_f64(g)[np.arange(N) // k]
    dense = np.einsum("ue,u,ui,eij->uj", onehot, alpha.astype(np.float64), gu, O.bf16_to_f64(W))
    logits = np.zeros((T, E), np.float32)
    for rho, cf in ((Fraction(1), Fraction(4)), (Fraction(1, 2), Fraction(5, 4))):
        st = O.route_stats(logits, idx, E, cf=cf, rho=rho)
        so, ids = O.select(O.score(g, phi, alpha, k), idx, E, st["quota"])
        dphi = O.grouped_dgrad(g, W, alpha, so, ids, E, k)
        rows = np.concatenate([dphi[e] for e in range(E)], axis=0)
        out = O.scatter_with_zeros(rows, ids, N)
        kept = np.zeros(N, dtype=bool)
        kept[ids] = True
        assert np.allclose(out[kept], dense[kept], rtol=1e-12, atol=1e-14)
        assert np.all(out[~kept] == 0.0)
        assert kept.sum() == st["retained"]
        if rho == 1:
            assert kept.all() and np.allclose(out, dense, rtol=1e-12, atol=1e-14)


def test_zero_masked_layout_gives_same_gradients():
    """Sec. 3.4: the zero-masked fixed-shape computation equals the compacted one."""
    T, k, E = 16, 2, 4
    g, phi, W, alpha, idx = _tiny(T=T, k=k, E=E, h=6, I=5, seed=4)
    st = O.route_stats(np.zeros((T, E), np.float32), idx, E, cf=Fraction(5, 4), rho=Fraction(1, 2))
    so, ids = O.select(O.score(g, phi, alpha, k), idx, E, st["quota"])
    dc, pc, _ = O.compact(g, phi, alpha, ids, k)
    dpad, ppad = O.compact_padded(dc, pc, so, E, st["C"])
    dW = O.grouped_wgrad_from_compact(dc, pc, so, E)
    dphi = O.grouped_dgrad_from_compact(dc, W, so, E)
    for e in range(E):
        D, P = O.bf16_to_f64(dpad[e]), O.bf16_to_f64(ppad[e])
        assert np.allclose(D.T @ P, dW[e], rtol=1e-13, atol=1e-15)
        full = D @ O.bf16_to_f64(W[e])
        q = so[e + 1] - so[e]
        assert np.allclose(full[:q], dphi[e], rtol=1e-13, atol=1e-15)
        assert np.all(full[q:] == 0)


def test_compacted_rows_reproduce_original_inputs_within_bf16():
    g, phi, W, alpha, idx = _tiny(T=10, k=2, E=3, h=16, I=8, seed=12)
    e_u = idx.reshape(-1)
    Q = np.bincount(e_u, minlength=3)
    so, ids = O.select(O.score(g, phi, alpha, 2), e_u, 3, Q)
    dc, pc, _ = O.compact(g, phi, alpha, ids, 2)
    a = O.grouped_wgrad(g, phi, alpha, so, ids, 3, 2)
    b = O.grouped_wgrad_from_compact(dc, pc, so, 3)
    for e in range(3):
        if np.any(a[e]):
            assert np.linalg.norm(a[e] - b[e]) <= 2 ** -8 * np.linalg.norm(a[e])


def test_aggregate_error_identity_and_bound():
    """Eq. (18)-(20): dropping D changes dW_e by -sum G_u; its squared norm is
    sum R_u plus twice the cross inner products, and at most (sum sqrt R)^2 <= d sum R."""
    T, k, E = 20, 2, 2
    g, phi, W, alpha, idx = _tiny(T=T, k=k, E=E, h=5, I=4, seed=21)
    e_u = idx.reshape(-1)
    n = np.bincount(e_u, minlength=E)
    R = O.score(g, phi, alpha, k)
    so_f, ids_f = O.select(R, e_u, E, n)
    Q = n - 3
    so_s, ids_s = O.select(R, e_u, E, Q)
    full = O.grouped_wgrad(g, phi, alpha, so_f, ids_f, E, k)
    part = O.grouped_wgrad(g, phi, alpha, so_s, ids_s, E, k)
    gf, pf = O.bf16_to_f64(g), O.bf16_to_f64(phi)
    for e in range(E):
        D = np.setdiff1d(np.flatnonzero(e_u == e), ids_s[so_s[e]:so_s[e + 1]])
        assert D.size == 3
        delta = part[e] - full[e]
        Gs = [np.outer(float(alpha[u]) * gf[u // k], pf[u]) for u in D]
        assert np.allclose(delta, -sum(Gs), rtol=1e-12, atol=1e-14)
        lhs = float(np.sum(delta * delta))
        cross = sum(float(np.sum(Gs[i] * Gs[j])) for i in range(3) for j in range(i + 1, 3))
        assert lhs == pytest.approx(float(R[D].sum()) + 2 * cross, rel=1e-10)
        assert lhs <= float(np.sqrt(R[D]).sum()) ** 2 * (1 + 1e-12)
        assert float(np.sqrt(R[D]).sum()) ** 2 <= D.size * float(R[D].sum()) * (1 + 1e-12)
        # the dropped pairs are the three smallest scores of the expert (Prop. 7.1)
        cand = np.flatnonzero(e_u == e)
        assert set(D.tolist()) == set(cand[np.lexsort((cand, R[cand]))][:3].tolist())


# ---------------------------------------------------------------------------
# generator sanity (a workload choice, not a result) and one full oracle pass


def test_generator_routing_shape_and_skew():
    w = get_workload("tiny_T256_E8_k2_h64_I32")
    inp = generate(w)
    assert inp.expert_idx.shape == (256, 2) and inp.g.shape == (256, 64) and inp.phi.shape == (512, 32)
    assert inp.W.shape == (8, 64, 32)
    a = inp.alpha.reshape(256, 2).astype(np.float64)
    assert np.allclose(a.sum(1), 1.0, atol=1e-6) and np.all(a[:, 0] >= a[:, 1])
    srt = np.sort(inp.expert_idx, axis=1)
    assert np.all(srt[:, 1:] != srt[:, :-1])


def test_stress_workload_has_empty_and_oversized_experts():
    from workloads.generate import routing

    w = get_workload("stress_T131072_E128_k8_h4096_I1408")
    logits, idx, alpha, bias, _ = routing(w)
    n = np.bincount(idx.reshape(-1), minlength=w.E)
    C = (w.cf.numerator * w.N) // (w.cf.denominator * w.E)
    assert (n == 0).sum() >= 1 and (n > C).sum() >= 1


def test_full_oracle_pass_on_tiny_workload():
    inp = generate("tiny_T256_E8_k2_h64_I32")
    out = O.backward_recalibration(inp)
    st = out["stats"]
    assert st["C"] == 80 and st["counts"].sum() == 512
    assert np.all(np.diff(out["sel_offsets"]) == st["quota"])
    assert out["delta_c"].shape == (st["retained"], 64)


# ---------------------------------------------------------------------------
# FC1 and its activation (LRMoE sec. 3.4: all four expert-backward GEMMs run on
# the retained rows; the activation is read as SwiGLU)


def test_swiglu_backward_matches_autograd_and_finite_differences():
    import torch

    rng = np.random.default_rng(41)
    ab = rng.standard_normal((7, 10)) * 2.0
    dphi = rng.standard_normal((7, 5))
    t_ab = torch.tensor(ab, dtype=torch.float64, requires_grad=True)
    a, b = t_ab[:, :5], t_ab[:, 5:]
    (torch.tensor(dphi) * (torch.nn.functional.silu(a) * b)).sum().backward()
    assert np.allclose(O.swiglu_backward(dphi, ab), t_ab.grad.numpy(), rtol=1e-12, atol=1e-14)
    assert np.allclose(O.swiglu_forward(ab), (torch.nn.functional.silu(a) * b).detach().numpy(), rtol=1e-14)
    # silu'(a) against a central difference of silu
    x = np.linspace(-8, 8, 33)
    h = 1e-6
    num = (O.silu(x + h) - O.silu(x - h)) / (2 * h)
    ana = O.swiglu_backward(np.ones((33, 1)), np.stack([x, np.ones(33)], axis=1))[:, 0]
    assert np.allclose(ana, num, rtol=1e-7, atol=1e-9)


def test_fc1_backward_equals_autograd_of_the_moe_layer():
    """The whole expert (FC1, SwiGLU, FC2, gate weight) for the retained pairs,
    differentiated by autograd, gives the FC1 weight gradient, the token input
    gradient (summed over the token's pairs) and the FC2 weight gradient of the
    oracle's path; dropped pairs contribute nothing."""
    import torch

    T, k, E, h, I = 10, 2, 3, 6, 4
    rng = np.random.default_rng(42)
    g, phi_unused, W2, alpha, idx = _tiny(T=T, k=k, E=E, h=h, I=I, seed=43)
    x_bits = f32_to_bf16_bits(rng.standard_normal((T, h)).astype(np.float32))
    W1_bits = f32_to_bf16_bits((rng.standard_normal((E, 2 * I, h)) * 0.3).astype(np.float32))
    x, W1 = O.bf16_to_f64(x_bits), O.bf16_to_f64(W1_bits)
    e_u = idx.reshape(-1)
    N = T * k
    ab = np.stack([W1[e_u[u]] @ x[u // k] for u in range(N)])
    for rho in (Fraction(1), Fraction(1, 2)):
        st = O.route_stats(np.zeros((T, E), np.float32), idx, E, cf=Fraction(4), rho=rho)
        R = O.score(g, f32_to_bf16_bits(O.swiglu_forward(ab).astype(np.float32)), alpha, k)
        so, ids = O.select(R, idx, E, st["quota"])
        dphi = O.grouped_dgrad(g, W2, alpha, so, ids, E, k)
        rows = np.concatenate([dphi[e] for e in range(E)], axis=0)
        dW1, dx_rows = O.fc1_backward(x, ab, W1, rows, so, ids, E, k)
        dx = O.combine_pairs(dx_rows, ids, T, k)
        # autograd of sum_t g_t . sum_{retained u of t} alpha_u W2_e silu(a_u) * b_u, [a_u; b_u] = W1_e x_t
        tx = torch.tensor(x, requires_grad=True)
        tW1 = torch.tensor(W1, requires_grad=True)
        tW2 = torch.tensor(O.bf16_to_f64(W2), requires_grad=True)
        tg = torch.tensor(O.bf16_to_f64(g))
        loss = torch.zeros((), dtype=torch.float64)
        for u in ids.tolist():
            t, e = u // k, int(e_u[u])
            abu = tW1[e] @ tx[t]
            phiu = torch.nn.functional.silu(abu[:I]) * abu[I:]
            loss = loss + float(alpha[u]) * (tg[t] @ (tW2[e] @ phiu))
        loss.backward()
        for e in range(E):
            assert np.allclose(dW1[e], tW1.grad[e].numpy(), rtol=1e-10, atol=1e-12)
        assert np.allclose(dx, tx.grad.numpy(), rtol=1e-10, atol=1e-12)
        kept = np.zeros(N, dtype=bool)
        kept[ids] = True
        if rho == 1:
            assert kept.all()
        else:
            assert not kept.all()


def test_combine_pairs_hand_case():
    rows = np.array([[1.0, 2.0], [10.0, 20.0], [100.0, 200.0]])
    out = O.combine_pairs(rows, [0, 1, 5], T=4, k=2)
    assert out.tolist() == [[11.0, 22.0], [0.0, 0.0], [100.0, 200.0], [0.0, 0.0]]
