"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties one oracle function to a hand-derived example, a closed form, a
library routine, an exact integral or an invariant that the pages or the
mathematics fix (Stochastic Sparse Attention for Memory-Bound Inference, paper
notes, Key designs 1-3).  A plausible slip anywhere in the oracle -- a threshold
off by one, the wrong side of a CDF boundary, a dropped 1/S, a wrong merge
weight, a transposed operand -- makes at least one of them fail.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from synthetic import float32_to_bf16_bits, bf16_bits_to_float32, generate, get_workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x):
    return bf16_bits_to_float32(float32_to_bf16_bits(np.asarray(x, dtype=np.float32))).astype(np.float64)


def _logit_problem(A, d):
    """q, K of head dim d whose logits are exactly log(A_i), so softmax(x) = A."""
    A = np.asarray(A, dtype=np.float64)
    q = np.zeros(d)
    q[0] = math.sqrt(d)
    K = np.zeros((A.size, d))
    K[:, 0] = np.log(A)
    return q, K


def _random_problem(rng, n, d, heavy=4, scale=6.0):
    q = _bf16(rng.standard_normal(d))
    K = rng.standard_normal((n, d))
    hot = rng.choice(n, size=min(heavy, n), replace=False)
    K[hot] += scale * q / np.linalg.norm(q) * math.sqrt(d) / 3.0
    return q, _bf16(K), _bf16(rng.standard_normal((n, d)))


def _numpy_softmax(q, K):
    """Independent softmax via numpy matmul + scipy (not the oracle's loops)."""
    from scipy.special import softmax

    return softmax((K @ q) / math.sqrt(K.shape[1]))


# ------------------------------------------------------------- hand examples


def test_hand_examples_from_golden():
    g = json.load(open(os.path.join(GOLDEN, "hand_examples.json")))
    V = np.asarray(g["V"], dtype=np.float64)
    q, K = _logit_problem(g["A"], V.shape[1])
    np.testing.assert_allclose(oracle.softmax(oracle.logits(q, K)), g["A"], rtol=1e-14)
    np.testing.assert_allclose(oracle.cdf(g["A"]), g["cdf"], rtol=1e-14)

    s = g["sys"]
    r = oracle.prop_head(q, K, V, s["S"], s["U"], s["tile"])
    assert r.J.tolist() == s["J"]
    assert r.counts.tolist() == s["counts"]
    np.testing.assert_allclose(r.mass, s["tile_mass"], rtol=1e-14)
    np.testing.assert_allclose(r.out, s["out"], atol=1e-15)

    f = g["flash"]
    r = oracle.flash_head(q, K, V, f["S"], f["U"], f["tile"])
    assert r.S_loc == f["S_loc"]
    assert r.J.tolist() == f["J"]
    np.testing.assert_allclose(r.weight, f["weight"], rtol=1e-14)
    np.testing.assert_allclose(r.out, f["out"], atol=1e-15)

    out, J = oracle.sampled_head("iid", q, K, V, g["iid"]["u"])
    assert J.tolist() == g["iid"]["J"]
    np.testing.assert_allclose(out, g["iid"]["out"], atol=1e-15)
    out, J = oracle.sampled_head("strat", q, K, V, g["strat"]["u"])
    assert J.tolist() == g["strat"]["J"]
    np.testing.assert_allclose(out, g["strat"]["out"], atol=1e-15)


def test_inverse_cdf_matches_linear_scan():
    """Smallest i with F(i) > t, including zero-mass keys and thresholds on boundaries."""
    rng = np.random.default_rng(7)
    for _ in range(200):
        n = int(rng.integers(1, 40))
        A = rng.random(n) * (rng.random(n) < 0.7)  # some zero-mass keys
        if A.sum() == 0:
            A[rng.integers(n)] = 1.0
        A /= A.sum()
        F = oracle.cdf(A)
        ts = np.concatenate([rng.random(20), F[:-1], [0.0]])
        for t in ts:
            if t >= 1.0:
                continue
            expect = int(np.argmax(F > t))
            assert oracle.inverse_cdf(F, t) == expect
            assert A[expect] > 0.0  # zero-mass keys are never chosen


# ------------------------------------------------------------- special cases


def test_one_hot_returns_that_row():
    """A one-hot A: every sample is that key, output is exactly V_j (prop and flash)."""
    rng = np.random.default_rng(1)
    n, d, j = 1000, 16, 613
    q = _bf16(rng.standard_normal(d))
    K = _bf16(rng.standard_normal((n, d)))
    K[j] = q * (1000.0 * math.sqrt(d) / float(q @ q))  # logit of key j = 1000
    V = _bf16(rng.standard_normal((n, d)))
    for S in (1, 16, 128, 1000):
        for U in (0.0, 0.5 / S, np.nextafter(1.0 / S, 0.0)):
            r = oracle.prop_head(q, K, V, S, U, tile=128)
            assert (r.J == j).all()
            assert np.array_equal(r.out, V[j])
            assert r.counts[j // 128] == S and r.counts.sum() == S
            f = oracle.flash_head(q, K, V, S, U, tile=128)
            assert np.array_equal(f.out, V[j])
            assert f.weight[j // 128] == 1.0


@pytest.mark.parametrize("n,tile", [(64, 16), (256, 64), (1024, 128)])
def test_uniform_with_S_equal_nk_is_the_mean(n, tile):
    """q = 0 gives A = 1/n; with S = n every key is drawn exactly once."""
    rng = np.random.default_rng(n)
    d = 8
    q = np.zeros(d)
    K = _bf16(rng.standard_normal((n, d)))
    V = _bf16(rng.standard_normal((n, d)))
    mean = V.sum(axis=0) / n  # exact: bf16 values, power-of-two n
    # (U is kept 0.001/n away from 1/n: closer, the float64 sum U + m/S rounds onto
    # the next CDF boundary m+1/n, which is rounding, not the sampler)
    for U in (0.0, 0.3 / n, 0.999 / n):
        r = oracle.prop_head(q, K, V, n, U, tile)
        assert r.J.tolist() == list(range(n))
        assert np.array_equal(r.out, mean)
        assert (r.counts == tile).all()
        # flash: S_loc = S / T = tile, so every tile draws each of its keys once
        f = oracle.flash_head(q, K, V, n, U, tile)
        assert f.S_loc == tile
        assert np.array_equal(np.sort(f.J.ravel()), np.arange(n))
        np.testing.assert_allclose(f.out, mean, rtol=0, atol=1e-15)


def test_flash_local_budget_closed_form():
    """S_loc = ceil(S / T) and the shared offset U * S / S_loc (ragged tail included)."""
    rng = np.random.default_rng(3)
    q, K, V = _random_problem(rng, 1000, 8)
    for S, tile in ((2048, 256), (16, 128), (7, 100), (1, 64)):
        T = -(-1000 // tile)
        f = oracle.flash_head(q, K, V, S, 0.0, tile)
        assert f.S_loc == -(-S // T)
        assert f.J.shape == (T, f.S_loc)
        for t in range(T):  # every sample stays inside its own tile
            assert ((f.J[t] >= t * tile) & (f.J[t] < min(1000, (t + 1) * tile))).all()


def test_empty_sequence_gives_zeros():
    q = np.ones(4)
    K = np.zeros((0, 4))
    r = oracle.prop_head(q, K, K, 8, 0.01, 16)
    assert np.array_equal(r.out, np.zeros(4)) and r.J.size == 0 and r.counts.size == 0
    assert np.array_equal(oracle.flash_head(q, K, K, 8, 0.01, 16).out, np.zeros(4))
    assert np.array_equal(oracle.exact_head(q, K, K), np.zeros(4))


# ------------------------------------------------------------- library routines


def test_exact_matches_torch_sdpa_float64():
    """Exact A V against torch's SDPA (default scale 1/sqrt(d)) in float64, with GQA."""
    rng = np.random.default_rng(11)
    B, Hq, Hkv, d = 2, 8, 2, 32
    lens = [300, 77]
    indptr = np.array([0, 300, 377])
    q = rng.standard_normal((B, Hq, d))
    k = rng.standard_normal((377, Hkv, d)) * 2.0
    v = rng.standard_normal((377, Hkv, d))
    res = oracle.run_problem("exact", q, k, v, indptr)
    G = Hq // Hkv
    for b in range(B):
        kb = torch.from_numpy(k[indptr[b] : indptr[b + 1]]).permute(1, 0, 2)  # [Hkv][n][d]
        vb = torch.from_numpy(v[indptr[b] : indptr[b + 1]]).permute(1, 0, 2)
        kb = kb.repeat_interleave(G, dim=0)[None]
        vb = vb.repeat_interleave(G, dim=0)[None]
        qb = torch.from_numpy(q[b])[None, :, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb)[0, :, 0, :].numpy()
        got = np.stack([res[(b, h)] for h in range(Hq)])
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    assert lens


def test_tile_masses_and_budget_bounds():
    """sum S_tile = S and |S_tile - S * Z_tile / Z| < 1 (systematic sampling),
    with Z_tile / Z taken from an independent numpy/scipy softmax."""
    rng = np.random.default_rng(5)
    for trial in range(30):
        n = int(rng.integers(1, 3000))
        d = int(rng.choice([8, 64]))
        tile = int(rng.choice([32, 128, 256]))
        S = int(rng.choice([1, 3, 16, 128, 4096]))
        q, K, V = _random_problem(rng, n, d, heavy=int(rng.integers(0, 9)), scale=float(rng.uniform(0, 12)))
        U = rng.random() / S
        r = oracle.prop_head(q, K, V, S, U, tile)
        A = _numpy_softmax(q, K)
        T = -(-n // tile)
        mass = np.array([A[t * tile : (t + 1) * tile].sum() for t in range(T)])
        np.testing.assert_allclose(r.mass, mass, rtol=1e-10, atol=1e-300)
        assert r.counts.sum() == S
        assert np.all(np.abs(r.counts - S * mass) < 1.0 + 1e-9)
        # the reducer's closed form: S_tile = N(C_t) - N(C_{t-1}), N(c) = ceil(S c - S U),
        # N(0) = 0 and N(1) = S, with C_t the inclusive prefix of the tile masses
        C = np.cumsum(mass)
        N = np.clip(np.ceil(S * C - S * U), 0, S).astype(np.int64)
        N[-1] = S
        closed = np.diff(np.concatenate([[0], N]))
        x = (S * C - S * U)[:-1]
        if np.all(np.abs(x - np.round(x)) > 1e-9):  # no threshold within rounding of a boundary
            assert closed.tolist() == r.counts.tolist()


# ------------------------------------------------------------- exact integration


def _sys_breakpoints(F, S):
    """U values in (0, 1/S) where some threshold U + m/S crosses a CDF value."""
    pts = [0.0, 1.0 / S]
    for f in F[:-1]:
        for m in range(S):
            u = f - m / S
            if 0.0 < u < 1.0 / S:
                pts.append(u)
    return np.unique(pts)


@pytest.mark.parametrize("seed", range(6))
def test_systematic_sampler_is_unbiased_exactly(seed):
    """E_U[estimate] = A V and E_U[#draws of key i] = S A_i, integrating exactly
    over the piecewise-constant dependence on U."""
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(1, 9))
    d = 3
    q, K, V = _random_problem(rng, n, d, heavy=1, scale=3.0)
    A = _numpy_softmax(q, K)
    exact = A @ V
    for S in (1, 2, 3, 4, 5, 8):
        F = oracle.cdf(A)
        pts = _sys_breakpoints(F, S)
        mean = np.zeros(d)
        draws = np.zeros(n)
        for a, b in zip(pts[:-1], pts[1:]):
            r = oracle.prop_head(q, K, V, S, 0.5 * (a + b), tile=4)
            w = (b - a) * S
            mean += w * r.out
            draws += w * np.bincount(r.J, minlength=n)
        np.testing.assert_allclose(mean, exact, rtol=0, atol=1e-12)
        np.testing.assert_allclose(draws, S * A, rtol=0, atol=1e-11)


@pytest.mark.parametrize("seed", range(6))
def test_flash_is_unbiased_exactly(seed):
    """E_U[flash estimate] = A V: per-tile systematic sampling with the shared offset
    U * S / S_loc, merged with weights Z_tile / Z."""
    rng = np.random.default_rng(200 + seed)
    n = int(rng.integers(2, 9))
    d = 3
    q, K, V = _random_problem(rng, n, d, heavy=1, scale=4.0)
    A = _numpy_softmax(q, K)
    exact = A @ V
    for S, tile in ((1, 2), (2, 3), (4, 2), (5, 4), (8, 3)):
        T = -(-n // tile)
        S_loc = -(-S // T)
        pts = [0.0, 1.0 / S]
        for t in range(T):
            At = A[t * tile : (t + 1) * tile]
            Ft = np.cumsum(At / At.sum())
            for f in Ft[:-1]:
                for m in range(S_loc):
                    u = (f - m / S_loc) * S_loc / S
                    if 0.0 < u < 1.0 / S:
                        pts.append(u)
        pts = np.unique(pts)
        mean = np.zeros(d)
        for a, b in zip(pts[:-1], pts[1:]):
            mean += (b - a) * S * oracle.flash_head(q, K, V, S, 0.5 * (a + b), tile).out
        np.testing.assert_allclose(mean, exact, rtol=0, atol=1e-12)


@pytest.mark.parametrize("mode", ["iid", "strat"])
def test_iid_and_stratified_are_unbiased_exactly(mode):
    """Integrate over u in [0,1)^S cell by cell.  For i.i.d. also check the
    closed-form variance (sum A V^2 - (A V)^2) / S."""
    rng = np.random.default_rng(300)
    for trial in range(4):
        n = int(rng.integers(1, 6))
        d = 2
        q, K, V = _random_problem(rng, n, d, heavy=1, scale=3.0)
        A = _numpy_softmax(q, K)
        F = oracle.cdf(A)
        exact = A @ V
        for S in (1, 2, 3):
            # breakpoints of each coordinate u_m
            cuts = []
            for m in range(S):
                if mode == "iid":
                    c = [f for f in F[:-1]]
                else:
                    c = [S * f - m for f in F[:-1] if 0.0 < S * f - m < 1.0]
                cuts.append(np.unique([0.0, 1.0] + c))
            mean = np.zeros(d)
            second = np.zeros(d)
            for cell in np.ndindex(*[len(c) - 1 for c in cuts]):
                lo = np.array([cuts[m][cell[m]] for m in range(S)])
                hi = np.array([cuts[m][cell[m] + 1] for m in range(S)])
                vol = float(np.prod(hi - lo))
                out, _ = oracle.sampled_head(mode, q, K, V, 0.5 * (lo + hi))
                mean += vol * out
                second += vol * out * out
            np.testing.assert_allclose(mean, exact, rtol=0, atol=1e-12)
            if mode == "iid":
                var = (A @ (V * V) - exact**2) / S
                np.testing.assert_allclose(second - mean**2, var, rtol=0, atol=1e-12)


# ------------------------------------------------------------- Monte Carlo


def test_monte_carlo_convergence_and_variance_ordering():
    """Mean over 4096 seeded offsets U is within 5 sigma of A V (sigma = sd/sqrt(4096));
    at small S the systematic sampler's variance is far below i.i.d. sampling's
    closed form, and it shrinks as S grows (the ordering of Table 2)."""
    rng = np.random.default_rng(42)
    n, d = 2048, 16
    q, K, V = _random_problem(rng, n, d, heavy=24, scale=5.0)
    A = _numpy_softmax(q, K)
    exact = A @ V
    iid_var = A @ (V * V) - exact**2
    prev = None
    for S in (16, 64):
        Us = rng.random(4096) / S
        est = np.stack([oracle.prop_head(q, K, V, S, U, 256, want_F=False).out for U in Us])
        sd = est.std(axis=0)
        assert np.all(np.abs(est.mean(axis=0) - exact) <= 5 * sd / math.sqrt(4096) + 1e-12)
        var = est.var(axis=0).sum()
        assert var < 0.5 * iid_var.sum() / S
        if prev is not None:
            assert var < prev
        prev = var


# ------------------------------------------------------------- page figures


def test_page_figures_and_llama8b_v_row_fraction():
    """The byte model and sample fractions the pages state, and the V-row bound
    (at most 4 S distinct rows per KV head, < 1.56% at 32k) on the synthetic
    Llama-3.1-8B layer."""
    g = json.load(open(os.path.join(GOLDEN, "paper_figures.json")))
    w = get_workload("llama8b_32k_b1")
    kv_bytes = 2 * w.num_kv_heads * w.length * w.head_dim * 2
    assert kv_bytes == g["kv_bytes_per_layer_per_token_32k_MB"]["value"] * 2**20
    assert w.group == g["gqa_group"]["value"]
    assert round(100 * w.S / w.length, 2) == g["prop_S128_fraction_of_nk_percent"]["value"]
    assert round(100 * 2048 / w.length, 2) == g["flash_S2048_fraction_of_nk_percent"]["value"]
    bound = g["prop_v_row_fraction_bound_percent"]["value"]
    assert math.floor(100 * 100 * w.group * w.S / w.length) / 100 == bound

    inp = generate(w)
    res = oracle.run_problem("prop", inp.q, inp.k_f32(), inp.v_f32(), inp.kv_indptr, S=w.S,
                             U=inp.U[0], tile=w.tile)
    for g_ in range(w.num_kv_heads):
        rows = set()
        for h in range(g_ * w.group, (g_ + 1) * w.group):
            rows.update(res[(0, h)].J.tolist())
        assert 100.0 * len(rows) / w.length < bound
    # every head concentrates on its planted keys: far fewer than S distinct rows
    assert max(len(set(r.J.tolist())) for r in res.values()) < w.S


# ------------------------------------------------------------------ Bernoulli q K^T
# "Stochastic Sparse Attention for Memory-Bound Inference" (paper notes), Key
# design 4: the ternary query drawn from q / max|q| estimates q K^T without bias;
# ablation table: the mean group query shares one feature set across a GQA group.


def _bernoulli_probs(q32: np.ndarray, group_mean: bool) -> np.ndarray:
    """The draw probabilities in single precision: [G][d] per head, [1][d] for the
    group mean (sum over heads in order, then / G)."""
    if group_mean:
        s = np.zeros(q32.shape[1], dtype=np.float32)
        for g in range(q32.shape[0]):
            s = (s + q32[g]).astype(np.float32)
        mean = (s / np.float32(q32.shape[0])).astype(np.float32)
        a = np.abs(mean)
        return (a / a.max()).astype(np.float32)[None, :]
    a = np.abs(q32)
    return (a / a.max(axis=1, keepdims=True)).astype(np.float32)


def _enumerate_draws(q32, draws, group_mean):
    """Every outcome of the Bernoulli draws with its probability, realised through
    uniforms (u = p/2 selects, u = (1+p)/2 does not); the oracle's c and read mask
    for each.  Yields (probability, c, read)."""
    import itertools

    p = _bernoulli_probs(q32, group_mean)  # [ns][d]
    ns, d = p.shape
    n = ns * draws * d
    pr = np.repeat(p[:, None, :], draws, axis=1).reshape(-1).astype(np.float64)
    for bits in itertools.product((0, 1), repeat=n):
        sel = np.array(bits, dtype=bool)
        prob = float(np.prod(np.where(sel, pr, 1.0 - pr)))
        if prob == 0.0:
            continue
        u = np.where(sel, pr / 2, (1.0 + pr) / 2).astype(np.float32).reshape(ns, draws, d)
        c, read = oracle.bernoulli_query(q32.astype(np.float64), u.astype(np.float64), group_mean)
        yield prob, c, read, p


@pytest.mark.parametrize("group_mean", [False, True])
@pytest.mark.parametrize("seed", [0, 1])
def test_bernoulli_query_is_unbiased_exactly(group_mean, seed):
    """E[c_g] = q_g for every head, by exact enumeration of all draw outcomes
    (d = 3, two draws; per head 2^12 outcomes, group mean 2^6), and the read
    probability of feature i is 1 - prod (1 - p)^draws over the draw sets."""
    rng = np.random.default_rng(seed)
    G, d, draws = 2, 3, 2
    q32 = rng.normal(size=(G, d)).astype(np.float32)
    Ec = np.zeros((G, d))
    Eread = np.zeros(d)
    total = 0.0
    p = None
    for prob, c, read, p in _enumerate_draws(q32, draws, group_mean):
        Ec += prob * c
        Eread += prob * read
        total += prob
    assert abs(total - 1.0) < 1e-12
    np.testing.assert_allclose(Ec, q32.astype(np.float64), rtol=1e-6, atol=1e-7)
    p64 = p.astype(np.float64)
    expect_read = 1.0 - np.prod((1.0 - p64) ** draws, axis=0)
    np.testing.assert_allclose(Eread, expect_read, rtol=1e-12, atol=1e-12)


def test_bernoulli_ternary_entries_and_monte_carlo():
    """Per head one draw gives a ternary query: c / max|q| in {-1, 0, +1} with the
    sign of q; over many draws the mean of c converges to q (5 sigma), and the
    read fraction to its expectation."""
    rng = np.random.default_rng(3)
    G, d = 1, 64
    q32 = rng.normal(size=(G, d)).astype(np.float32)
    mx = float(np.abs(q32).max())
    c, read = oracle.bernoulli_query(q32.astype(np.float64), rng.random((1, 1, d)), False)
    t = c[0] / mx
    assert set(np.unique(t)).issubset({-1.0, 0.0, 1.0})
    assert np.all((t == 0) | (np.sign(t) == np.sign(q32[0])))
    assert np.array_equal(read, t != 0)
    n = 4000
    acc = np.zeros(d)
    sq = np.zeros(d)
    nread = 0
    for _ in range(n):
        c, read = oracle.bernoulli_query(q32.astype(np.float64), rng.random((1, 1, d)), False)
        acc += c[0]
        sq += c[0] ** 2
        nread += read.sum()
    mean = acc / n
    sd = np.sqrt(np.maximum(sq / n - mean ** 2, 1e-30) / n)
    assert np.all(np.abs(mean - q32[0]) < 5 * sd + 1e-9)
    p = np.abs(q32[0]).astype(np.float64) / mx
    assert abs(nread / (n * d) - p.mean()) < 5 * np.sqrt(p.mean() * (1 - p.mean()) / (n * d)) + 1e-3


@pytest.mark.parametrize("group_mean", [False, True])
def test_bernoulli_with_all_probabilities_one_is_the_exact_query(group_mean):
    """|q_i| all equal (and, for the group mean, equal heads): every p = 1, every
    feature is read, c = q whatever the uniforms, and the prop head on c is the
    prop head on q."""
    rng = np.random.default_rng(5)
    G, d, n = 2, 16, 300
    row = np.where(rng.random(d) < 0.5, -0.75, 0.75).astype(np.float32)
    q32 = np.stack([row, row if group_mean else -row])
    ns = 1 if group_mean else G
    c, read = oracle.bernoulli_query(q32.astype(np.float64), rng.random((ns, 3, d)), group_mean)
    assert read.all()
    np.testing.assert_array_equal(c, q32.astype(np.float64))
    K = rng.normal(size=(n, d))
    V = rng.normal(size=(n, d))
    a = oracle.prop_head(c[0], K, V, 16, 0.01, 64)
    b = oracle.prop_head(q32[0].astype(np.float64), K, V, 16, 0.01, 64)
    np.testing.assert_array_equal(a.J, b.J)
    np.testing.assert_array_equal(a.out, b.out)


def test_mean_group_query_shares_one_feature_set():
    """Mean group query: the read mask is the selection of the one shared draw
    set, whatever the heads; per head, the union over heads (never smaller for
    the same uniforms of head 0 when the heads are equal)."""
    rng = np.random.default_rng(9)
    G, d = 4, 32
    q32 = rng.normal(size=(G, d)).astype(np.float32)
    u = rng.random((1, 2, d))
    c, read = oracle.bernoulli_query(q32.astype(np.float64), u, True)
    p = _bernoulli_probs(q32, True)[0]
    sel = (u.astype(np.float32) < p).any(axis=(0, 1))
    assert np.array_equal(read, sel)
    assert np.array_equal(c != 0, np.broadcast_to(sel, c.shape) & (q32 != 0))
