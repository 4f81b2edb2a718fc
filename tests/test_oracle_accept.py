"""Pins of the fp64 speculative-acceptance oracle.

"How speculative decoding doubles LLM speed" (section "Absolute mathematical
exactness") fixes what the rejection sampler must produce: every emitted
token is distributed exactly as the target distribution p, the first draft
is accepted with probability alpha = sum min(p, q), and the draft
distribution q cancels out.  These are checked statistically (chi-squared,
binomial) on a 16-token vocabulary, plus the deterministic corner cases."""
import numpy as np
import pytest
import scipy.special
import scipy.stats

from spec_verify_paged_gb300 import workloads as W

V, K = 16, 3
TRIALS = 200_000
P_MIN = 1e-3


def _rows(seed, noise=0.7):
    rng = np.random.default_rng(seed)
    t = (rng.standard_normal((K + 1, V)) * 1.5).astype(np.float32)
    d = (t[:K] + rng.standard_normal((K, V)) * noise).astype(np.float32)
    return t, d


def _trials(oracle_mod, t, d, seed, n=TRIALS, tokens=None, u=None):
    """n independent acceptance runs over the same logit rows, with draft
    tokens drawn from q = softmax(d) and fresh uniforms."""
    rng = np.random.default_rng(seed)
    q = scipy.special.softmax(d.astype(np.float64), axis=-1)
    if tokens is None:
        tokens = np.stack([rng.choice(V, size=n, p=q[i]) for i in range(K)],
                          axis=1).astype(np.int32)
    if u is None:
        u = W.uniforms01(rng, (n, K + 1))
    tl = np.broadcast_to(t, (n, K + 1, V))
    dl = np.broadcast_to(d, (n, K, V))
    res = oracle_mod.spec_accept(tl, dl, tokens, u)
    return res, tokens, u


def _chi2_p(samples, p):
    counts = np.bincount(samples, minlength=V).astype(np.float64)
    expect = p * counts.sum()
    keep = expect > 0
    assert counts[~keep].sum() == 0, "a token of zero probability was emitted"
    return scipy.stats.chisquare(counts[keep], expect[keep]).pvalue


def test_emitted_tokens_follow_the_target(oracle_mod):
    """Lossless identity: P(emit x) = min(p, q) + max(0, p - q) = p(x) at
    every position, whatever q is."""
    t, d = _rows(1)
    res, _, _ = _trials(oracle_mod, t, d, seed=2)
    p = scipy.special.softmax(t.astype(np.float64), axis=-1)
    out, nacc = res["out_tokens"], res["n_accepted"]
    assert _chi2_p(out[:, 0], p[0]) > P_MIN
    sel = nacc >= 1                      # position 2 exists
    assert _chi2_p(out[sel, 1], p[1]) > P_MIN
    sel = nacc >= 2
    assert _chi2_p(out[sel, 2], p[2]) > P_MIN
    sel = nacc == K                      # the bonus token
    assert sel.sum() > 1000
    assert _chi2_p(out[sel, K], p[K]) > P_MIN
    # shape of the output: n_accepted + 1 tokens, then -1 padding
    n_out = (out >= 0).sum(axis=1)
    assert np.array_equal(n_out, nacc + 1)
    for k in range(K + 1):
        assert np.all(out[n_out <= k, k] == -1)


def test_first_acceptance_rate_is_alpha(oracle_mod):
    """Rejection mass 1 - alpha = sum max(0, p - q), alpha = sum min(p, q)."""
    t, d = _rows(3, noise=1.2)
    res, _, _ = _trials(oracle_mod, t, d, seed=4)
    p = scipy.special.softmax(t[0].astype(np.float64))
    q = scipy.special.softmax(d[0].astype(np.float64))
    alpha = np.minimum(p, q).sum()
    rate = (res["n_accepted"] >= 1).mean()
    sd = np.sqrt(alpha * (1 - alpha) / TRIALS)
    assert abs(rate - alpha) < 4.5 * sd
    assert 0.2 < alpha < 0.95  # the test is informative


def test_identical_draft_accepts_everything(oracle_mod):
    """q = p: the ratio is exactly 1, every draft is accepted and the bonus
    comes from the last target row."""
    t, _ = _rows(5)
    res, tokens, _ = _trials(oracle_mod, t, t[:K].copy(), seed=6, n=50_000)
    assert np.all(res["n_accepted"] == K)
    assert np.array_equal(res["out_tokens"][:, :K], tokens)
    p = scipy.special.softmax(t[K].astype(np.float64))
    assert _chi2_p(res["out_tokens"][:, K], p) > P_MIN


def test_impossible_draft_is_always_rejected(oracle_mod):
    """q concentrated on a token x with p(x) = 0: every draft is rejected at
    the first position, and the residual max(0, p - q) is p itself on the
    other tokens, so the replacement follows p."""
    t, d = _rows(7)
    x = 5
    t = t.copy()
    d = np.zeros_like(d)
    t[0, x] = -1.0e4                 # exp underflows: p(x) == 0 exactly
    d[0, x] = 60.0                   # q(x) ~ 1, q(y) ~ e^-60
    n = 60_000
    rng = np.random.default_rng(8)
    u = W.uniforms01(rng, (n, K + 1))
    u[:, 0] = np.maximum(u[:, 0], np.float32(2.0 ** -24))   # r > 0
    tokens = np.full((n, K), x, np.int32)
    res, _, _ = _trials(oracle_mod, t, d, seed=8, n=n, tokens=tokens, u=u)
    assert np.all(res["n_accepted"] == 0)
    assert np.all(res["out_tokens"][:, 1:] == -1)
    p = scipy.special.softmax(t[0].astype(np.float64))
    assert _chi2_p(res["out_tokens"][:, 0], p) > P_MIN


def test_inverse_cdf_ends(oracle_mod):
    """Inverse CDF in token order: u = 0 picks the first token of positive
    weight; u just below 1 picks the last one."""
    t, _ = _rows(9)
    d = t[:K].copy()                 # all accepted -> bonus from p_K
    tok = np.zeros((2, K), np.int32)
    u = np.array([[0.5] * K + [0.0], [0.5] * K + [1 - 2.0 ** -24]], np.float32)
    res, _, _ = _trials(oracle_mod, t, d, 0, n=2, tokens=tok, u=u)
    assert res["out_tokens"][0, K] == 0
    assert res["out_tokens"][1, K] == V - 1
    # a residual with leading zero weights: first positive entry wins at u=0
    t2 = t.copy()
    d2 = t[:K].copy()
    d2[0, :4] += 5.0                 # q > p on tokens 0..3 -> w = 0 there
    tok2 = np.full((1, K), 0, np.int32)
    u2 = np.array([[0.999999] + [0.5] * (K - 1) + [0.0]], np.float32)
    res2, _, _ = _trials(oracle_mod, t2, d2, 0, n=1, tokens=tok2, u=u2)
    assert res2["n_accepted"][0] == 0
    assert res2["out_tokens"][0, 0] == 4


def test_boundary_draws_are_flagged(oracle_mod):
    """q = p gives ratio 1; r = 1 - 2^-24 lies within 1e-6 of it."""
    t, _ = _rows(11)
    tok = np.zeros((2, K), np.int32)
    u = np.array([[1 - 2.0 ** -24] + [0.5] * K, [0.5] * (K + 1)], np.float32)
    res, _, _ = _trials(oracle_mod, t, t[:K].copy(), 0, n=2, tokens=tok, u=u)
    assert res["near_boundary"][0] == 1
    assert np.all(res["n_accepted"] == K)


def test_bad_draft_token_is_reported(oracle_mod):
    t, d = _rows(13)
    tok = np.array([[0, V, 1]], np.int32)
    with pytest.raises(ValueError):
        _trials(oracle_mod, t, d, 0, n=1, tokens=tok)


def test_accept_workload_generator(oracle_mod):
    """The verify-gqa acceptance workload runs through the oracle and draws
    a spread of acceptance counts."""
    wl = W.make_accept(batch=64, num_draft=4, vocab=32000, seed=3)
    res = oracle_mod.spec_accept(wl.target_logits, wl.draft_logits,
                                 wl.draft_tokens, wl.uniforms)
    assert set(np.unique(res["n_accepted"])) >= {0, 4}
    assert (res["out_tokens"] >= 0).sum() == (res["n_accepted"] + 1).sum()
