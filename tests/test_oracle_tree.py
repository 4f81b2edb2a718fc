"""Pins of the fp64 draft-tree oracle (attention mask and tree acceptance).

"How speculative decoding doubles LLM speed" (section "Modern architecture
variants") describes SpecInfer: the draft is a tree of several branches,
verified in one pass with a two-dimensional attention mask; "Speculative
decoding: how AI models get faster without getting bigger" adds that the
verifier keeps the longest accepted path.  The pins: a chain-shaped tree
is the causal verify block; every tree node attends exactly like a plain
sequence made of the prefix and its root path (torch SDPA in fp64); on a
chain the tree acceptance is the linear rule; and the emitted token
follows the target distribution whatever the branching (chi-squared on a
16-token vocabulary)."""
import math

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

from helpers import widen
from spec_verify_paged_gb300 import workloads as W

P_MIN = 1e-3


def _chain_mask(B, n):
    return np.tile(np.array([(2 << i) - 1 for i in range(n)], np.uint32), (B, 1))


def test_tree_mask_helper():
    par = W.binary_tree_parents(2)
    assert par.tolist() == [-1, 0, 0, 1, 1, 2, 2]
    m = W.tree_mask_from_parents(par)
    # node 5: path 0 -> 2 -> 5
    assert m[5] == (1 << 0) | (1 << 2) | (1 << 5)
    assert np.array_equal(W.tree_mask_from_parents(np.arange(-1, 5)),
                          _chain_mask(1, 6)[0])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chain_tree_is_the_causal_block(oracle_mod, dtype):
    """A tree whose node i has parent i-1 is the linear draft: the mask
    must reproduce the causal verify block exactly."""
    cfg = W.small_config(batch=3, num_q_heads=8, num_kv_heads=2, head_dim=64,
                         q_len=6, dtype=dtype, ctx_min=6, ctx_max=80, seed=21)
    wl = W.make_attention(cfg)
    o1, l1 = oracle_mod.paged_attention(wl.q, wl.k_cache, wl.v_cache,
                                        wl.block_table, wl.seq_lens, 6, 0, 0,
                                        wl.scale)
    o2, l2 = oracle_mod.paged_tree_attention(wl.q, wl.k_cache, wl.v_cache,
                                             wl.block_table, wl.seq_lens, 6,
                                             _chain_mask(3, 6), wl.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def _logical_kv(wl, b, g, L):
    """Rows 0..L-1 of (b, g) gathered from the paged cache by hand."""
    D = wl.k_cache.shape[-1]
    K = np.zeros((L, D))
    V = np.zeros((L, D))
    for j in range(L):
        blk = wl.block_table[b, j // W.BLOCK_SIZE]
        K[j] = widen(wl.k_cache[blk, g, j % W.BLOCK_SIZE])
        V[j] = widen(wl.v_cache[blk, g, j % W.BLOCK_SIZE])
    return K, V


def test_tree_node_attends_like_its_root_path(oracle_mod):
    """Node i of the tree sees the cached prefix and the nodes on its path
    from the root: its output is plain softmax attention over exactly that
    key sequence (torch SDPA in fp64, keys gathered by hand)."""
    depth = 2
    n = (1 << (depth + 1)) - 1
    cfg = W.small_config(batch=2, num_q_heads=4, num_kv_heads=2, head_dim=64,
                         q_len=n, dtype="bf16", ctx_min=n + 1, ctx_max=70,
                         seed=22)
    wl = W.make_attention(cfg)
    par = W.binary_tree_parents(depth)
    mask = np.tile(W.tree_mask_from_parents(par), (2, 1))
    out, lse = oracle_mod.paged_tree_attention(
        wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.seq_lens, n, mask,
        wl.scale)
    G = cfg.num_q_heads // cfg.num_kv_heads
    for b in range(2):
        L = int(wl.seq_lens[b])
        base = L - n
        for i in range(n):
            path = []
            c = i
            while c >= 0:
                path.append(c)
                c = par[c]
            keys = list(range(base)) + [base + c for c in sorted(path)]
            for h in range(cfg.num_q_heads):
                K, V = _logical_kv(wl, b, h // G, L)
                Kt = torch.from_numpy(K[keys])[None, None]
                Vt = torch.from_numpy(V[keys])[None, None]
                Qt = torch.from_numpy(widen(wl.q[b, i, h]))[None, None, None]
                ref = torch.nn.functional.scaled_dot_product_attention(
                    Qt, Kt, Vt, scale=float(wl.scale))[0, 0, 0].numpy()
                np.testing.assert_allclose(out[b, i, h], ref, rtol=0, atol=1e-12)
                s = float(wl.scale) * (K[keys] @ widen(wl.q[b, i, h]))
                assert abs(lse[b, i, h] - scipy.special.logsumexp(s)) < 1e-12


def test_tree_mask_rejects_window(oracle_mod):
    """The tree mask carries no sink/window policy: the entry point takes
    none, and the shared core refuses the combination."""
    cfg = W.small_config(batch=1, num_q_heads=2, num_kv_heads=1, head_dim=64,
                         q_len=3, dtype="f32", ctx_min=20, ctx_max=20, seed=1)
    wl = W.make_attention(cfg)
    bad = _chain_mask(1, 3)
    bad[0, 0] = 0  # a node that sees no new key at all is still allowed
    oracle_mod.paged_tree_attention(wl.q, wl.k_cache, wl.v_cache,
                                    wl.block_table, wl.seq_lens, 3, bad,
                                    wl.scale)


# --------------------------------------------------------------------------
# tree acceptance
# --------------------------------------------------------------------------

def test_chain_tree_accept_is_the_linear_rule(oracle_mod):
    """Node i+1 hangs below node i: tree acceptance must make the linear
    decisions (u of node i+1 = u_i of the linear rule, u of the root =
    the linear rule's draw uniform u_K)."""
    K, V, B = 4, 1000, 400
    lin = W.make_accept(batch=B, num_draft=K, vocab=V, seed=31)
    N = K + 1
    par = np.tile(np.arange(-1, K, dtype=np.int32), (B, 1))
    tok = np.concatenate([np.full((B, 1), -1, np.int32), lin.draft_tokens], 1)
    draft = np.concatenate([lin.draft_logits, lin.target_logits[:, K:]], 1)
    u = np.concatenate([lin.uniforms[:, K:], lin.uniforms[:, :K]], 1)
    tr = oracle_mod.spec_accept_tree(lin.target_logits, draft, par, tok, u)
    ref = oracle_mod.spec_accept(lin.target_logits, lin.draft_logits,
                                 lin.draft_tokens, lin.uniforms)
    ok = (tr["near_boundary"] == 0) & (ref["near_boundary"] == 0)
    assert ok.mean() > 0.8
    assert np.array_equal(tr["n_accepted"][ok], ref["n_accepted"][ok])
    assert np.array_equal(tr["out_tokens"][ok], ref["out_tokens"][ok])
    # accepted path nodes are 1 .. n_accepted
    for b in np.nonzero(ok)[0][:50]:
        n = tr["n_accepted"][b]
        assert tr["out_nodes"][b, :n].tolist() == list(range(1, n + 1))
        assert np.all(tr["out_nodes"][b, n:] == -1)
    assert len(np.unique(tr["n_accepted"])) == K + 1


def _fixed_tree_trials(par, seed, n, Vv=16, noise=0.9):
    """n acceptance runs over the same tree shape and logit rows; each
    node's children drawn independently from q = softmax(draft row)."""
    rng = np.random.default_rng(seed)
    N = len(par)
    t = (rng.standard_normal((N, Vv)) * 1.5).astype(np.float32)
    d = (t + rng.standard_normal((N, Vv)) * noise).astype(np.float32)
    q = scipy.special.softmax(d.astype(np.float64), axis=-1)
    tok = np.full((n, N), -1, np.int32)
    for c in range(1, N):
        tok[:, c] = rng.choice(Vv, size=n, p=q[par[c]])
    u = W.uniforms01(rng, (n, N))
    tl = np.broadcast_to(t, (n, N, Vv))
    dl = np.broadcast_to(d, (n, N, Vv))
    pa = np.broadcast_to(np.asarray(par, np.int32), (n, N))
    return t, d, tok, u, tl, dl, pa


def _chi2_p(samples, p):
    counts = np.bincount(samples, minlength=p.size).astype(np.float64)
    expect = p * counts.sum()
    keep = expect > 0
    assert counts[~keep].sum() == 0, "a token of zero probability was emitted"
    return scipy.stats.chisquare(counts[keep], expect[keep]).pvalue


@pytest.mark.parametrize("par", [[-1, 0, 0, 0], [-1, 0, 0, 1, 1, 2, 2]])
def test_tree_accept_emits_the_target_distribution(oracle_mod, par):
    """"Absolute mathematical exactness" for a tree: with the children of a
    node drawn independently from q, trying them in turn with the residual
    carried between them leaves the first emitted token distributed as p of
    the root (and, after an accepted child, the next one as p of that
    child)."""
    n = 200_000
    t, d, tok, u, tl, dl, pa = _fixed_tree_trials(par, seed=len(par), n=n)
    res = oracle_mod.spec_accept_tree(tl, dl, pa, tok, u)
    p = scipy.special.softmax(t.astype(np.float64), axis=-1)
    out = res["out_tokens"]
    assert _chi2_p(out[:, 0], p[0]) > P_MIN
    nodes = res["out_nodes"]
    for c in range(1, len(par)):
        if any(par[k] == c for k in range(len(par))):
            sel = nodes[:, 0] == c          # first step accepted child c
            if sel.sum() > 5000:
                assert _chi2_p(out[sel, 1], p[c]) > P_MIN
    # the path is a root path: each accepted node's parent is the previous
    nacc = res["n_accepted"]
    for b in range(200):
        prev = 0
        for k in range(nacc[b]):
            assert par[nodes[b, k]] == prev
            prev = nodes[b, k]
    # several children make rejection rarer than a single one would
    assert (nacc >= 1).mean() > 0.5


def test_identical_draft_follows_first_children(oracle_mod):
    """q = p at every node: the first child is always accepted, so the path
    is 1, 3, 7 in a depth-3 binary tree and the bonus comes from the leaf."""
    wl = W.make_tree_accept(batch=64, depth=3, vocab=500, seed=33)
    draft = wl.target_logits.copy()
    res = oracle_mod.spec_accept_tree(wl.target_logits, draft, wl.parents,
                                      wl.node_tokens, wl.uniforms)
    assert np.all(res["n_accepted"] == 3)
    assert np.all(res["out_nodes"][:, :3] == np.array([1, 3, 7]))
    assert np.array_equal(res["out_tokens"][:, :3], wl.node_tokens[:, [1, 3, 7]])


def test_malformed_tree_and_bad_token_are_reported(oracle_mod):
    wl = W.make_tree_accept(batch=2, depth=1, vocab=50, seed=34)
    bad = wl.parents.copy()
    bad[1, 2] = 2                       # a node below itself
    with pytest.raises(ValueError):
        oracle_mod.spec_accept_tree(wl.target_logits, wl.draft_logits, bad,
                                    wl.node_tokens, wl.uniforms)
    tok = wl.node_tokens.copy()
    tok[0, 1] = 50
    with pytest.raises(ValueError):
        oracle_mod.spec_accept_tree(wl.target_logits, wl.draft_logits,
                                    wl.parents, tok, wl.uniforms)
