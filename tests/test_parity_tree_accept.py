"""GPU tree acceptance vs the fp64 oracle.

Accepted paths, their nodes and the drawn tokens must be identical given the
same uniforms.  Where the oracle reports a decision within 1e-6 of its
boundary, the GPU outcome must be one of the outcomes the oracle lists as
reachable when such comparisons may go either way
(oracle.spec_accept_tree_valid); those sequences are counted."""
import numpy as np
import pytest

from helpers import compare_tree_accept, to_dev
from spec_verify_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def svp():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import spec_verify_paged_gb300 as m
    return m


def _gpu(svp, wl):
    import torch
    toks, nodes, nacc = svp.spec_accept_tree(
        to_dev(wl.target_logits), to_dev(wl.draft_logits), to_dev(wl.parents),
        to_dev(wl.node_tokens), to_dev(wl.uniforms))
    torch.cuda.synchronize()
    return toks.cpu().numpy(), nodes.cpu().numpy(), nacc.cpu().numpy()


def _check(svp, oracle_mod, wl, max_boundary_frac=0.15):
    toks, nodes, nacc = _gpu(svp, wl)
    ref = oracle_mod.spec_accept_tree(wl.target_logits, wl.draft_logits,
                                      wl.parents, wl.node_tokens, wl.uniforms)
    valid = oracle_mod.spec_accept_tree_valid(wl.target_logits,
                                              wl.draft_logits, wl.parents,
                                              wl.node_tokens, wl.uniforms)
    nb, _ = compare_tree_accept(toks, nodes, nacc, ref, valid, wl.node_tokens)
    assert nb <= max(2, max_boundary_frac * len(nacc)), nb
    assert svp.read_device_status() == 0
    return nacc


def test_tree_verify_workload(svp, oracle_mod):
    """16 sequences, a 15-node binary draft tree, vocab 32000."""
    wl = W.make_tree_accept(**W.TREE_ACCEPT_CONFIG)
    _check(svp, oracle_mod, wl)


@pytest.mark.parametrize("depth,V,seed", [(3, 32000, 1), (2, 5000, 2),
                                          (1, 1001, 3), (3, 50257, 4)])
def test_many_sequences(svp, oracle_mod, depth, V, seed):
    wl = W.make_tree_accept(batch=256, depth=depth, vocab=V, seed=50 + seed)
    nacc = _check(svp, oracle_mod, wl, max_boundary_frac=0.3)
    assert len(np.unique(nacc)) >= 2


@pytest.mark.parametrize("shape", ["star", "random", "chain"])
def test_tree_shapes(svp, oracle_mod, shape):
    """A root with 15 children (up to 14 residual passes at one node), a
    random tree per sequence, and a 16-node chain."""
    rng = np.random.default_rng(7)
    B, N, V = 128, 16, 2048
    if shape == "star":
        par = np.array([-1] + [0] * (N - 1), np.int32)
        wl = W.make_tree_accept(batch=B, vocab=V, seed=61, parents=par,
                                noise_std=1.5)
    elif shape == "chain":
        par = np.arange(-1, N - 1, dtype=np.int32)
        wl = W.make_tree_accept(batch=B, vocab=V, seed=62, parents=par)
    else:
        wl = W.make_tree_accept(batch=B, vocab=V, seed=63,
                                parents=W.binary_tree_parents(3)[:N - 1])
        for b in range(B):  # re-hang nodes at random, keep tokens valid
            wl.parents[b, 1:] = [int(rng.integers(0, c)) for c in range(1, N - 1)]
    _check(svp, oracle_mod, wl, max_boundary_frac=0.3)


def test_chain_tree_matches_linear_kernel(svp):
    """On a chain the tree call makes exactly the linear call's decisions
    (uniforms reordered: node i+1 <- u_i, root <- u_K)."""
    import torch
    K, V, B = 4, 32000, 64
    lin = W.make_accept(batch=B, num_draft=K, vocab=V, seed=71)
    par = np.tile(np.arange(-1, K, dtype=np.int32), (B, 1))
    tok = np.concatenate([np.full((B, 1), -1, np.int32), lin.draft_tokens], 1)
    draft = np.concatenate([lin.draft_logits, lin.target_logits[:, K:]], 1)
    u = np.concatenate([lin.uniforms[:, K:], lin.uniforms[:, :K]], 1)
    t1, n1, a1 = svp.spec_accept_tree(to_dev(lin.target_logits), to_dev(draft),
                                      to_dev(par), to_dev(tok), to_dev(u))
    t2, a2 = svp.spec_accept(to_dev(lin.target_logits), to_dev(lin.draft_logits),
                             to_dev(lin.draft_tokens), to_dev(lin.uniforms))
    torch.cuda.synchronize()
    assert np.array_equal(a1.cpu().numpy(), a2.cpu().numpy())
    assert np.array_equal(t1.cpu().numpy(), t2.cpu().numpy())


def test_identical_draft_follows_first_children(svp, oracle_mod):
    wl = W.make_tree_accept(batch=32, depth=3, vocab=4000, seed=72)
    wl.draft_logits[:] = wl.target_logits
    toks, nodes, nacc = _gpu(svp, wl)
    assert np.all(nacc == 3)
    assert np.all(nodes[:, :3] == np.array([1, 3, 7]))


def test_bad_tree_is_flagged(svp):
    wl = W.make_tree_accept(batch=4, depth=2, vocab=1000, seed=73)
    wl.parents[1, 3] = 5          # a parent after its child
    wl.node_tokens[2, 4] = 1000   # a token outside the vocabulary
    toks, nodes, nacc = _gpu(svp, wl)
    assert nacc[1] == -1 and nacc[2] == -1
    assert np.all(toks[[1, 2]] == -1) and np.all(nodes[[1, 2]] == -1)
    assert np.all(nacc[[0, 3]] >= 0)
    assert svp.read_device_status() & 4
