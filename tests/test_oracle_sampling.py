"""Pins of the oracle's sampling pieces: Philox known answers, inverse-CDF draws,
the exact output distribution of speculative rejection sampling (Leviathan et al.:
it equals the target distribution), and SPD-vs-AR agreement in distribution at T>0."""
import os

import numpy as np
import pytest
from scipy import stats

import spd_inputs as si
from oracle import Model, SPDOracle, ar_decode, philox
from oracle.sampling import inverse_cdf, probs, residual, verify_exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_philox_known_answers():
    n = 0
    for line in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        w = [int(x, 16) for x in line.split()]
        assert philox.philox4x32_10(w[0:4], w[4:6]) == tuple(w[6:10])
        n += 1
    assert n == 3


def test_philox_uniforms_are_uniform():
    u = np.array([philox.uniform(12345, t, p) for t in range(2000) for p in range(5)])
    assert u.min() >= 0.0 and u.max() < 1.0
    counts, _ = np.histogram(u, bins=20, range=(0, 1))
    assert stats.chisquare(counts).pvalue > 1e-3
    assert philox.uniform(1, 5, 2) == philox.u24(1, 5, 2) / 2.0 ** 24


def test_inverse_cdf_intervals():
    w = np.array([0.1, 0.0, 0.2, 0.3, 0.4])
    c = np.cumsum(w)
    for u in np.linspace(0, 0.999999, 1001):
        i = inverse_cdf(w, u)
        assert w[i] > 0
        assert (c[i - 1] if i else 0.0) <= u * c[-1] < c[i]
    # unnormalised weights pick the same indices
    assert inverse_cdf(3 * w, 0.55) == inverse_cdf(w, 0.55) == 3


@pytest.mark.parametrize("seed", range(6))
def test_rejection_sampling_preserves_target_exactly(seed):
    rng = np.random.default_rng(seed)
    V = 2 + seed
    pT = rng.dirichlet(np.ones(V) * 0.5)
    pD = rng.dirichlet(np.ones(V) * 0.5)
    np.testing.assert_allclose(verify_exact(pT, pD), pT, atol=1e-13)


def test_rejection_sampling_special_cases():
    p = np.array([0.2, 0.3, 0.5])
    np.testing.assert_allclose(verify_exact(p, p), p, atol=1e-15)       # always kept
    pT, pD = np.array([0.0, 1.0, 0.0]), np.array([0.5, 0.0, 0.5])        # disjoint support
    np.testing.assert_allclose(residual(pT, pD), pT)
    np.testing.assert_allclose(verify_exact(pT, pD), pT, atol=1e-15)


def test_probs_is_softmax_over_temperature():
    z = np.array([1.0, 2.0, 3.0])
    e = np.exp(z / 0.5)
    np.testing.assert_allclose(probs(z, 0.5), e / e.sum(), rtol=1e-14)


def _exact_ar_marginals(m, prompt, T, k):
    """Exact distribution of the first k generated tokens by enumeration (V small)."""
    V = m.dm.V
    from itertools import product
    dist = {}
    for seq in product(range(V), repeat=k):
        kv = m.new_cache(32)
        H = m.target_layers(m.embed[list(prompt)], 0, kv, 0, m.dm.L)
        h, pos, pr = H[-1], len(prompt), 1.0
        for j, y in enumerate(seq):
            pr *= probs(m.logits(h), T)[y]
            if j + 1 < k:
                h = m.target_layers(m.embed[[y]], pos, kv, 0, m.dm.L)[0]
                pos += 1
        dist[seq] = pr
    return dist


def test_spd_sampling_matches_ar_distribution():
    """At T>0 the SPD token stream has the target's distribution (rejection sampling is
    lossless): chi-square of 1500 seeded SPD runs against the exact AR law of the
    first 3 generated tokens on a 4-token vocabulary."""
    dm = si.ModelDims(L=4, d=16, Hq=2, Hkv=1, hd=8, F=32, V=4, dtype="fp32")
    anchors = (0, 2, 4)
    m = Model(dm, si.make_target(dm, 8, norms="perturbed"), si.make_pdm(dm, 1, 3, 8, norms="perturbed"), anchors)
    # scale logits up so the laws are far from uniform and drafts are often rejected
    m.lm_head = m.lm_head * 40.0
    prompt, T, k = [1, 3, 0], 1.0, 3
    exact = _exact_ar_marginals(m, prompt, T, k)
    runs = 1500
    counts = {}
    rejects = 0
    for s in range(runs):
        o = SPDOracle(m, 2, 32, temperature=T, seed=1000 + s)
        toks = tuple(o.run(prompt, k))
        counts[toks] = counts.get(toks, 0) + 1
        rejects += o.stats()["rejects"]
    keys = sorted(exact)
    obs = np.array([counts.get(q, 0) for q in keys], dtype=float)
    exp = np.array([exact[q] for q in keys]) * runs
    big = exp >= 5
    obs_c = np.append(obs[big], obs[~big].sum())
    exp_c = np.append(exp[big], exp[~big].sum())
    assert rejects > 100
    assert stats.chisquare(obs_c, exp_c).pvalue > 1e-3
