"""GPU verify epilogue (temperature, token mask, greedy) vs the fp64 oracle.

Sampling: tokens and counts identical, except that where the oracle places a
decision within 1e-6 of its boundary the GPU outcome must be one of the
outcomes the oracle lists as reachable when such comparisons may go either
way (oracle.spec_accept_valid).  Greedy: identical."""
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


def _pack(allowed):
    """bool [B, R, V] -> uint32 [B, R, ceil(V/32)], bit x%32 of word x/32."""
    B, R, V = allowed.shape
    words = (V + 31) // 32
    pad = np.zeros((B, R, words * 32), bool)
    pad[..., :V] = allowed
    return np.packbits(pad, axis=-1, bitorder="little").view(np.uint32).copy()


def _workload(B, K, V, seed, T=1.0, density=None, greedy_hits=0.0):
    wl = W.make_accept(batch=B, num_draft=K, vocab=V, seed=seed)
    rng = np.random.default_rng(seed + 1000)
    allowed = None
    if density is not None:
        allowed = rng.random((B, K + 1, V)) < density
        allowed[..., 0] = True
    # drafts drawn from the tempered, masked draft distribution
    logits = wl.draft_logits.astype(np.float64) / T
    if allowed is not None:
        logits = np.where(allowed[:, :K], logits, -np.inf)
    wl.draft_tokens = np.argmax(logits + rng.gumbel(size=logits.shape),
                                axis=-1).astype(np.int32)
    if greedy_hits > 0:
        t = wl.target_logits[:, :K].astype(np.float64)
        if allowed is not None:
            t = np.where(allowed[:, :K], t, -np.inf)
        am = np.argmax(t, axis=-1).astype(np.int32)
        hit = rng.random(am.shape) < greedy_hits
        wl.draft_tokens[hit] = am[hit]
    return wl, allowed


def _check(svp, oracle_mod, wl, allowed, T=1.0, greedy=False,
           max_boundary_frac=0.3):
    import torch
    bits = None if allowed is None else _pack(allowed)
    toks, nacc = svp.spec_accept(
        to_dev(wl.target_logits), to_dev(wl.draft_logits),
        to_dev(wl.draft_tokens), to_dev(wl.uniforms), temperature=T,
        allowed=None if bits is None else to_dev(bits.view(np.int32)),
        greedy=greedy)
    torch.cuda.synchronize()
    toks, nacc = toks.cpu().numpy(), nacc.cpu().numpy()
    ref = oracle_mod.spec_accept_ex(wl.target_logits, wl.draft_logits,
                                    wl.draft_tokens, wl.uniforms,
                                    temperature=T, allowed=bits, greedy=greedy)
    if greedy:  # no boundary: argmax ties go to the smallest index
        assert np.array_equal(nacc, ref["n_accepted"])
        assert np.array_equal(toks, ref["out_tokens"])
    else:
        valid = oracle_mod.spec_accept_valid(
            wl.target_logits, wl.draft_logits, wl.draft_tokens, wl.uniforms,
            temperature=T, allowed=bits)
        nb, _ = compare_accept(toks, nacc, ref, valid, wl.draft_tokens,
                               label="spec_accept_ex")
        assert nb <= max(2, max_boundary_frac * len(nacc))
    assert svp.read_device_status() == 0
    if allowed is not None:  # every emitted token is allowed at its position
        B, K1 = toks.shape
        for b in range(B):
            for i in range(K1):
                if toks[b, i] >= 0:
                    assert allowed[b, i, toks[b, i]]
    return nacc


@pytest.mark.parametrize("T", [0.6, 1.7])
def test_temperature(svp, oracle_mod, T):
    wl, _ = _workload(64, 4, 32000, 91, T=T)
    nacc = _check(svp, oracle_mod, wl, None, T=T)
    assert len(np.unique(nacc)) >= 3


@pytest.mark.parametrize("V,density", [(32000, 0.5), (5003, 0.3), (4096, 0.02)])
def test_token_mask(svp, oracle_mod, V, density):
    """Aligned and odd vocabularies (bulk and plain staging), dense and
    very sparse masks."""
    wl, allowed = _workload(48, 4, V, 92 + V, density=density)
    _check(svp, oracle_mod, wl, allowed)


def test_mask_with_temperature_many_sequences(svp, oracle_mod):
    """512 sequences: more clusters than fit at once (8-CTA clusters)."""
    wl, allowed = _workload(512, 3, 2000, 93, T=0.8, density=0.7)
    _check(svp, oracle_mod, wl, allowed, T=0.8)


def test_excluded_draft_is_rejected(svp, oracle_mod):
    wl, allowed = _workload(32, 4, 1000, 94, density=0.5)
    for b in range(32):          # draft 0 points at an excluded token
        x = int(np.nonzero(~allowed[b, 0])[0][0])
        wl.draft_tokens[b, 0] = x
    wl.uniforms[:, 0] = 0.0
    nacc = _check(svp, oracle_mod, wl, allowed)
    assert np.all(nacc == 0)


@pytest.mark.parametrize("masked", [False, True])
@pytest.mark.parametrize("V", [32000, 777])
def test_greedy(svp, oracle_mod, masked, V):
    wl, allowed = _workload(96, 4, V, 95 + V, density=0.5 if masked else None,
                            greedy_hits=0.8)
    nacc = _check(svp, oracle_mod, wl, allowed, greedy=True)
    assert len(np.unique(nacc)) >= 3


@pytest.mark.parametrize("greedy", [False, True])
def test_token_mask_with_a_staging_ring(svp, oracle_mod, greedy):
    """15 drafts over vocab 32,000: 31 rows (16 for greedy) of 2,000-token
    slices do not fit the 72 KB staging area, so pass 1 streams them through
    a ring of slots refilled piece by piece while the mask rewrites staged
    values; tokens and counts match the oracle."""
    wl, allowed = _workload(8, 15, 32000, 96 + int(greedy), T=0.9, density=0.6,
                            greedy_hits=0.9 if greedy else 0.0)
    _check(svp, oracle_mod, wl, allowed, T=0.9 if not greedy else 1.0,
           greedy=greedy)
