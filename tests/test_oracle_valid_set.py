"""Pins of the oracle's valid-outcome sets near a decision boundary.

The acceptance rule ("How speculative decoding doubles LLM speed", step 3)
is a chain of comparisons of the uniforms against the rule's quantities.
Decisions within eps of their boundary are not compared exactly; the
functions under test list the outcomes the rule can reach when each such
comparison may go either way.  They are pinned to the plain oracle
functions (themselves pinned by chi-squared and the corner cases):

* with eps = 0 the set is exactly the rule's single outcome;
* a sequence that the plain oracle does not flag has exactly its outcome;
* moving every uniform by less than eps and running the plain rule always
  lands inside the set (so the set is large enough), and over many such
  moves the outcomes reached cover the set (so it is not larger than the
  band allows).
"""
import numpy as np
import pytest

from helpers import accept_in_valid_set, tree_accept_in_valid_set
from spec_verify_paged_gb300 import workloads as W


def _linear_outcome(res, b):
    j = int(res["n_accepted"][b])
    return (j, int(res["out_tokens"][b, j]))


def _valid_linear(v, b):
    """{(j, token)} of one sequence's valid set."""
    out = set()
    K1 = v["path_valid"].shape[1]
    for j in range(K1):
        if v["path_valid"][b, j]:
            n = int(v["n_cand"][b, j])
            assert n <= v["cand"].shape[2]
            out |= {(j, int(t)) for t in v["cand"][b, j, :n]}
    return out


def _perturbed(u, eps, rng, n_random):
    """u [K+1] moved by the axis extremes (+-0.99 eps on one entry) and by
    n_random random vectors with entries in (-0.99 eps, 0.99 eps), kept in
    [0, 1)."""
    K1 = u.size
    moves = [np.zeros(K1)]
    for i in range(K1):
        for s in (-0.99, -0.5, 0.5, 0.99):
            m = np.zeros(K1)
            m[i] = s * eps
            moves.append(m)
    moves += list(rng.uniform(-0.99 * eps, 0.99 * eps, size=(n_random, K1)))
    uu = np.clip(u[None, :].astype(np.float64) + np.array(moves), 0.0,
                 1.0 - 2.0 ** -24).astype(np.float32)
    return uu


@pytest.mark.parametrize("temperature,masked", [(1.0, False), (0.6, True)])
def test_zero_band_is_the_rule_itself(oracle_mod, temperature, masked):
    wl = W.make_accept(batch=200, num_draft=4, vocab=500, seed=71)
    allowed = None
    if masked:
        rng = np.random.default_rng(3)
        allowed = rng.integers(0, 2**32, size=(200, 5, (500 + 31) // 32),
                               dtype=np.uint64).astype(np.uint32)
    ref = oracle_mod.spec_accept_ex(wl.target_logits, wl.draft_logits,
                                    wl.draft_tokens, wl.uniforms,
                                    temperature=temperature, allowed=allowed)
    v = oracle_mod.spec_accept_valid(wl.target_logits, wl.draft_logits,
                                     wl.draft_tokens, wl.uniforms,
                                     temperature=temperature, allowed=allowed,
                                     eps=0.0)
    for b in range(200):
        assert _valid_linear(v, b) == {_linear_outcome(ref, b)}, b
    ok = accept_in_valid_set(ref["out_tokens"], ref["n_accepted"],
                             wl.draft_tokens, v)
    assert ok.all()


def test_unflagged_sequences_have_one_outcome(oracle_mod):
    wl = W.make_accept(batch=256, num_draft=4, vocab=32000, seed=72)
    ref = oracle_mod.spec_accept(wl.target_logits, wl.draft_logits,
                                 wl.draft_tokens, wl.uniforms)
    v = oracle_mod.spec_accept_valid(wl.target_logits, wl.draft_logits,
                                     wl.draft_tokens, wl.uniforms)
    flagged = 0
    for b in range(256):
        s = _valid_linear(v, b)
        assert _linear_outcome(ref, b) in s
        if ref["near_boundary"][b] == 0:
            assert s == {_linear_outcome(ref, b)}, b
        else:
            flagged += 1
            assert len(s) >= 1
    # about 2e-6 per token of positive weight: a few percent of sequences
    assert flagged < 0.2 * 256


@pytest.mark.parametrize("temperature,masked", [(1.0, False), (0.7, True)])
def test_moves_within_the_band_stay_in_the_set_and_cover_it(
        oracle_mod, temperature, masked):
    """A wide band (eps = 0.02) on a 16-token vocabulary, so that many
    sequences have a comparison inside it."""
    eps, B, K, V = 0.02, 120, 3, 16
    wl = W.make_accept(batch=B, num_draft=K, vocab=V, seed=73)
    rng = np.random.default_rng(5)
    allowed = None
    if masked:
        bits = rng.random((B, K + 1, V)) < 0.8
        bits[..., 0] = True
        pad = np.zeros((B, K + 1, 32), bool)
        pad[..., :V] = bits
        allowed = np.packbits(pad, axis=-1, bitorder="little").view(np.uint32)
    v = oracle_mod.spec_accept_valid(wl.target_logits, wl.draft_logits,
                                     wl.draft_tokens, wl.uniforms,
                                     temperature=temperature, allowed=allowed,
                                     eps=eps)
    covered = multi = 0
    for b in range(B):
        valid = _valid_linear(v, b)
        uu = _perturbed(wl.uniforms[b], eps, rng, 1500)
        n = uu.shape[0]
        rep = lambda a: np.broadcast_to(a[b], (n,) + a.shape[1:])  # noqa: E731
        res = oracle_mod.spec_accept_ex(
            rep(wl.target_logits), rep(wl.draft_logits), rep(wl.draft_tokens),
            uu, temperature=temperature,
            allowed=None if allowed is None else rep(allowed))
        reached = {_linear_outcome(res, i) for i in range(n)}
        assert reached <= valid, (b, reached - valid)
        covered += reached == valid
        multi += len(valid) > 1
    assert multi >= 20            # the band is exercised
    assert covered >= 0.9 * B     # and rarely holds an outcome no move reached


def test_tree_zero_band_and_unflagged(oracle_mod):
    par = W.binary_tree_parents(3)
    wl = W.make_tree_accept(batch=64, vocab=2000, seed=74, parents=par)
    ref = oracle_mod.spec_accept_tree(wl.target_logits, wl.draft_logits,
                                      wl.parents, wl.node_tokens, wl.uniforms)
    for eps in (0.0, 1e-6):
        v = oracle_mod.spec_accept_tree_valid(
            wl.target_logits, wl.draft_logits, wl.parents, wl.node_tokens,
            wl.uniforms, eps=eps)
        ok = tree_accept_in_valid_set(ref["out_tokens"], ref["out_nodes"],
                                      ref["n_accepted"], wl.node_tokens, v)
        assert ok.all()
        for b in range(64):
            if eps == 0.0 or ref["near_boundary"][b] == 0:
                assert v[b]["n_outcomes"] == 1
                assert v[b]["outcomes"][0]["n_cand"] == 1


@pytest.mark.parametrize("depth", [1, 2])
def test_tree_moves_within_the_band_stay_in_the_set_and_cover_it(oracle_mod,
                                                                 depth):
    eps, B, V = 0.02, 60, 16
    par = W.binary_tree_parents(depth)
    wl = W.make_tree_accept(batch=B, vocab=V, seed=75 + depth, parents=par)
    v = oracle_mod.spec_accept_tree_valid(wl.target_logits, wl.draft_logits,
                                          wl.parents, wl.node_tokens,
                                          wl.uniforms, eps=eps)
    rng = np.random.default_rng(6)
    covered = multi = 0
    for b in range(B):
        valid = {(o["nodes"], c) for o in v[b]["outcomes"] for c in o["cand"]}
        assert v[b]["n_outcomes"] == len(v[b]["outcomes"])
        uu = _perturbed(wl.uniforms[b], eps, rng, 1500)
        n = uu.shape[0]
        rep = lambda a: np.broadcast_to(a[b], (n,) + a.shape[1:])  # noqa: E731
        res = oracle_mod.spec_accept_tree(rep(wl.target_logits),
                                          rep(wl.draft_logits), rep(wl.parents),
                                          rep(wl.node_tokens), uu)
        reached = set()
        for i in range(n):
            k = int(res["n_accepted"][i])
            reached.add((tuple(int(x) for x in res["out_nodes"][i, :k]),
                         int(res["out_tokens"][i, k])))
        assert reached <= valid, (b, reached - valid)
        covered += reached == valid
        multi += len(valid) > 1
    assert multi >= 10
    assert covered >= 0.9 * B


def test_membership_helper_rejects_wrong_outcomes(oracle_mod):
    """The comparison helper itself: a wrong count, a wrong draft copy, a
    token outside the candidates or a missing -1 pad each fail."""
    wl = W.make_accept(batch=32, num_draft=4, vocab=300, seed=76)
    ref = oracle_mod.spec_accept(wl.target_logits, wl.draft_logits,
                                 wl.draft_tokens, wl.uniforms)
    v = oracle_mod.spec_accept_valid(wl.target_logits, wl.draft_logits,
                                     wl.draft_tokens, wl.uniforms, eps=0.0)
    toks, nacc = ref["out_tokens"].copy(), ref["n_accepted"].copy()
    assert accept_in_valid_set(toks, nacc, wl.draft_tokens, v).all()
    b = int(np.argmax(nacc < 4))         # a sequence with a rejection
    j = int(nacc[b])
    t2 = toks.copy()
    t2[b, j] = (t2[b, j] + 1) % 300
    assert not accept_in_valid_set(t2, nacc, wl.draft_tokens, v)[b]
    n2 = nacc.copy()
    n2[b] = j + 1
    assert not accept_in_valid_set(toks, n2, wl.draft_tokens, v)[b]
    t3 = toks.copy()
    t3[b, 4] = 7 if j < 4 else t3[b, 4]
    if j < 4:
        assert not accept_in_valid_set(t3, nacc, wl.draft_tokens, v)[b]
    b2 = int(np.argmax(nacc > 0))        # a sequence with an accepted draft
    t4 = toks.copy()
    t4[b2, 0] = (t4[b2, 0] + 1) % 300
    assert not accept_in_valid_set(t4, nacc, wl.draft_tokens, v)[b2]


def test_excluded_draft_at_zero_uniform_has_only_the_rejection(oracle_mod):
    """A draft token the mask excludes has p(x) = 0: it is rejected even at
    u = 0, on every band (the comparison is not near a boundary)."""
    B, K, V = 40, 3, 64
    wl = W.make_accept(batch=B, num_draft=K, vocab=V, seed=77)
    allowed = np.full((B, K + 1, 2), 0xFFFFFFFF, np.uint32)
    x = wl.draft_tokens[:, 0]
    allowed[np.arange(B), 0, x >> 5] &= ~(np.uint32(1) << (x & 31).astype(np.uint32))
    wl.uniforms[:, 0] = 0.0
    for eps in (0.0, 1e-6, 0.05):
        v = oracle_mod.spec_accept_valid(wl.target_logits, wl.draft_logits,
                                         wl.draft_tokens, wl.uniforms,
                                         allowed=allowed, eps=eps)
        assert v["path_valid"][:, 0].all()
        assert not v["path_valid"][:, 1:].any()
