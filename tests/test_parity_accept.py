"""GPU spec_accept vs the fp64 oracle.

Accept counts and output tokens must be identical given the same uniforms.
Where the oracle reports a decision within 1e-6 of its boundary, either
answer of that comparison is correct: the GPU outcome must then be one of
the outcomes the oracle lists as reachable (oracle.spec_accept_valid).
Flagged sequences are counted and reported."""
import numpy as np
import pytest

from helpers import compare_accept, to_dev
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
    toks, nacc = svp.spec_accept(to_dev(wl.target_logits),
                                 to_dev(wl.draft_logits),
                                 to_dev(wl.draft_tokens), to_dev(wl.uniforms))
    torch.cuda.synchronize()
    return toks.cpu().numpy(), nacc.cpu().numpy()


def _check(svp, oracle_mod, wl, max_boundary_frac=0.15):
    """Exact agreement on every sequence whose decisions all lie farther
    than 1e-6 from their boundary; valid-set membership on the others.  The
    flagged share is about 2e-6 x (tokens of positive weight) for the draw,
    i.e. a few percent at vocab 32000, and is only bounded loosely."""
    toks, nacc = _gpu(svp, wl)
    ref = oracle_mod.spec_accept(wl.target_logits, wl.draft_logits,
                                 wl.draft_tokens, wl.uniforms)
    valid = oracle_mod.spec_accept_valid(wl.target_logits, wl.draft_logits,
                                         wl.draft_tokens, wl.uniforms)
    n_boundary, _ = compare_accept(toks, nacc, ref, valid, wl.draft_tokens)
    assert n_boundary <= max(2, max_boundary_frac * len(nacc)), n_boundary
    assert svp.read_device_status() == 0
    return n_boundary, nacc


def test_verify_workload_accept(svp, oracle_mod):
    """verify-gqa acceptance: 16 sequences, K = 4, vocab 32000."""
    wl = W.make_accept(**W.ACCEPT_CONFIG)
    _check(svp, oracle_mod, wl)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_many_sequences(svp, oracle_mod, seed):
    wl = W.make_accept(batch=512, num_draft=4, vocab=32000, seed=100 + seed)
    nb, nacc = _check(svp, oracle_mod, wl)
    assert len(np.unique(nacc)) == 5   # every acceptance count occurs


@pytest.mark.parametrize("K,V", [(1, 2), (3, 16), (7, 1000), (3, 1001),
                                 (15, 4096), (4, 50257), (2, 151936)])
def test_shapes(svp, oracle_mod, K, V):
    """Odd vocabularies (not a multiple of 4: unstaged path), tiny ones
    (empty slices), large K and large V."""
    wl = W.make_accept(batch=64, num_draft=K, vocab=V, seed=K * 7 + V)
    _check(svp, oracle_mod, wl, max_boundary_frac=0.3)


def test_identical_draft_accepts_all(svp, oracle_mod):
    wl = W.make_accept(batch=64, num_draft=4, vocab=32000, seed=9)
    wl.draft_logits[:] = wl.target_logits[:, :4]
    _, nacc = _check(svp, oracle_mod, wl)
    assert np.all(nacc == 4)


def test_impossible_draft_always_rejected(svp, oracle_mod):
    wl = W.make_accept(batch=64, num_draft=3, vocab=5000, seed=10)
    x = 123
    wl.draft_tokens[:, 0] = x
    wl.target_logits[:, 0, x] = -1.0e4
    wl.draft_logits[:, 0, :] = 0.0
    wl.draft_logits[:, 0, x] = 60.0
    wl.uniforms[:, 0] = np.maximum(wl.uniforms[:, 0], np.float32(2.0 ** -24))
    _, nacc = _check(svp, oracle_mod, wl)
    assert np.all(nacc == 0)


def test_bad_token_is_flagged(svp):
    import torch
    wl = W.make_accept(batch=4, num_draft=4, vocab=1000, seed=11)
    wl.draft_tokens[2, 3] = 1000
    toks, nacc = _gpu(svp, wl)
    assert nacc[2] == -1 and np.all(toks[2] == -1)
    assert np.all(nacc[[0, 1, 3]] >= 0)
    assert svp.read_device_status() & 4


def test_empty_batch(svp):
    import torch
    z = torch.zeros((0, 5, 100), dtype=torch.float32, device="cuda:0")
    d = torch.zeros((0, 4, 100), dtype=torch.float32, device="cuda:0")
    t = torch.zeros((0, 4), dtype=torch.int32, device="cuda:0")
    u = torch.zeros((0, 5), dtype=torch.float32, device="cuda:0")
    toks, nacc = svp.spec_accept(z, d, t, u)
    assert toks.shape == (0, 5) and nacc.shape == (0,)
