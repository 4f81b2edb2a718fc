"""Pins of the verify-epilogue oracle: temperature, constrained decoding
mask, greedy verification.

"How speculative decoding doubles LLM speed" (section "Deployment limits")
names sampling temperature; "How Moondream cut VLM inference latency"
(section "Mechanism two: forward first, then sample") sets the logits of
tokens the grammar does not allow to -inf before sampling.  Pins: emitted
tokens follow softmax(target / T) (scipy, chi-squared); excluded tokens are
never emitted and the rest follow the renormalised target; greedy
verification matches numpy's argmax; trivial options reproduce the plain
rule."""
import numpy as np
import pytest
import scipy.special
import scipy.stats

from spec_verify_paged_gb300 import workloads as W

V, K = 16, 3
P_MIN = 1e-3


def _rows(seed, noise=0.8):
    rng = np.random.default_rng(seed)
    t = (rng.standard_normal((K + 1, V)) * 1.5).astype(np.float32)
    d = (t[:K] + rng.standard_normal((K, V)) * noise).astype(np.float32)
    return t, d


def _trials(t, d, seed, n, T=1.0, allowed_rows=None):
    """n runs over the same rows; drafts drawn from the tempered, masked q."""
    rng = np.random.default_rng(seed)
    logits = d.astype(np.float64) / T
    if allowed_rows is not None:
        logits = np.where(allowed_rows[:K], logits, -np.inf)
    q = scipy.special.softmax(logits, axis=-1)
    tokens = np.stack([rng.choice(V, size=n, p=q[i]) for i in range(K)],
                      axis=1).astype(np.int32)
    u = W.uniforms01(rng, (n, K + 1))
    return (np.broadcast_to(t, (n, K + 1, V)), np.broadcast_to(d, (n, K, V)),
            tokens, u)


def _chi2_p(samples, p):
    counts = np.bincount(samples, minlength=V).astype(np.float64)
    expect = p * counts.sum()
    keep = expect > 0
    assert counts[~keep].sum() == 0, "a token of zero probability was emitted"
    return scipy.stats.chisquare(counts[keep], expect[keep]).pvalue


def _bits(allowed_rows, B):
    """[K+1, V] bool -> [B, K+1, ceil(V/32)] uint32 masks."""
    words = (V + 31) // 32
    m = np.zeros((K + 1, words), np.uint32)
    for i in range(K + 1):
        for x in np.nonzero(allowed_rows[i])[0]:
            m[i, x >> 5] |= np.uint32(1 << (x & 31))
    return np.broadcast_to(m, (B, K + 1, words))


def test_trivial_options_are_the_plain_rule(oracle_mod):
    wl = W.make_accept(batch=300, num_draft=4, vocab=777, seed=81)
    words = (777 + 31) // 32
    full = np.full((300, 5, words), 0xFFFFFFFF, np.uint32)
    a = oracle_mod.spec_accept(wl.target_logits, wl.draft_logits,
                               wl.draft_tokens, wl.uniforms)
    b = oracle_mod.spec_accept_ex(wl.target_logits, wl.draft_logits,
                                  wl.draft_tokens, wl.uniforms, 1.0, full)
    assert np.array_equal(a["out_tokens"], b["out_tokens"])
    assert np.array_equal(a["n_accepted"], b["n_accepted"])


@pytest.mark.parametrize("T", [0.5, 2.0])
def test_temperature_sets_the_emitted_distribution(oracle_mod, T):
    """Both models at temperature T: every emitted token follows
    softmax(target / T) (scipy), whatever the draft does."""
    t, d = _rows(82)
    n = 150_000
    tl, dl, tok, u = _trials(t, d, 83, n, T=T)
    res = oracle_mod.spec_accept_ex(tl, dl, tok, u, temperature=T)
    p = scipy.special.softmax(t.astype(np.float64) / T, axis=-1)
    out, nacc = res["out_tokens"], res["n_accepted"]
    assert _chi2_p(out[:, 0], p[0]) > P_MIN
    sel = nacc >= 1
    assert _chi2_p(out[sel, 1], p[1]) > P_MIN
    # and not the untempered target
    p1 = scipy.special.softmax(t[0].astype(np.float64))
    assert _chi2_p(out[:, 0], p1) < 1e-6


def test_mask_excludes_tokens_and_renormalises(oracle_mod):
    """Tokens outside the allowed set are never emitted; the allowed ones
    follow the target softmax restricted to them."""
    rng = np.random.default_rng(84)
    allowed = rng.random((K + 1, V)) < 0.6
    allowed[:, 0] = True
    t, d = _rows(85)
    n = 150_000
    tl, dl, tok, u = _trials(t, d, 86, n, allowed_rows=allowed)
    res = oracle_mod.spec_accept_ex(tl, dl, tok, u, allowed=_bits(allowed, n))
    out, nacc = res["out_tokens"], res["n_accepted"]
    for i in range(K + 1):
        sel = nacc >= i if i > 0 else np.ones(n, bool)
        col = out[sel, i]
        col = col[col >= 0]
        assert np.all(allowed[i][col])
        p = scipy.special.softmax(np.where(allowed[i], t[i].astype(np.float64),
                                           -np.inf))
        if col.size > 5000:
            assert _chi2_p(col, p) > P_MIN


def test_excluded_draft_token_is_rejected(oracle_mod):
    t, d = _rows(87)
    allowed = np.ones((K + 1, V), bool)
    allowed[0, 3] = False
    n = 1000
    tok = np.full((n, K), 3, np.int32)
    u = np.zeros((n, K + 1), np.float32)  # u = 0 would accept any ratio >= 0
    res = oracle_mod.spec_accept_ex(np.broadcast_to(t, (n, K + 1, V)),
                                    np.broadcast_to(d, (n, K, V)), tok, u,
                                    allowed=_bits(allowed, n))
    assert np.all(res["n_accepted"] == 0)
    assert np.all(res["out_tokens"][:, 0] != 3)


def test_greedy_is_argmax_verification(oracle_mod):
    """Greedy: accept while the draft equals numpy's argmax of the target
    row (over allowed tokens), then emit that argmax."""
    wl = W.make_accept(batch=400, num_draft=4, vocab=300, seed=88)
    rng = np.random.default_rng(89)
    am = np.argmax(wl.target_logits, axis=-1)          # [B, K+1]
    tok = wl.draft_tokens.copy()
    take = rng.random(tok.shape) < 0.7                  # many drafts correct
    tok[take] = am[:, :4][take]
    res = oracle_mod.spec_accept_ex(wl.target_logits, wl.draft_logits, tok,
                                    wl.uniforms, greedy=True)
    for b in range(400):
        j = 0
        while j < 4 and tok[b, j] == am[b, j]:
            j += 1
        assert res["n_accepted"][b] == j
        assert list(res["out_tokens"][b, :j]) == list(tok[b, :j])
        assert res["out_tokens"][b, j] == am[b, j]
    # with a mask the argmax is over the allowed tokens only
    words = (300 + 31) // 32
    allowed = np.full((400, 5, words), 0xFFFFFFFF, np.uint32)
    for b in range(400):       # exclude every row's unrestricted argmax
        for i in range(5):
            allowed[b, i, am[b, i] >> 5] &= ~np.uint32(1 << (am[b, i] & 31))
    res2 = oracle_mod.spec_accept_ex(wl.target_logits, wl.draft_logits, tok,
                                     wl.uniforms, greedy=True, allowed=allowed)
    second = np.argsort(-wl.target_logits, axis=-1, kind="stable")[:, :, 1]
    for b in range(400):
        j = res2["n_accepted"][b]
        assert res2["out_tokens"][b, j] == second[b, j]
        assert res2["out_tokens"][b, j] != am[b, j]
