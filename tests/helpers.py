"""Shared test helpers: storage widening and simple layout builders.

Nothing here computes attention or acceptance; the helpers only widen stored
bits to float64 and rearrange pages (labels of physical blocks are arbitrary,
so permuting them together with the table must not change any result).
"""
import numpy as np

from spec_verify_paged_gb300 import workloads as W


def widen(a):
    """Stored values (fp32 or bf16 bits) as float64."""
    if a.dtype == np.uint16:
        return W.bf16_bits_to_f32(a).astype(np.float64)
    return a.astype(np.float64)


def identity_layout(rng, B, Hkv, D, L, dtype="f32", Hq=None, q_len=1):
    """Sequences of equal length L stored contiguously: sequence b owns
    physical blocks b*nblk .. b*nblk+nblk-1 in order, so the logical K of
    (b, g) is simply k_cache[b*nblk:(b+1)*nblk, g].reshape(-1, D)[:L]."""
    Hq = Hq or Hkv
    nblk = -(-L // W.BLOCK_SIZE)
    shape = (B * nblk, Hkv, W.BLOCK_SIZE, D)
    k = W._normals(rng, shape, dtype)
    v = W._normals(rng, shape, dtype)
    q = W._normals(rng, (B, q_len, Hq, D), dtype)
    table = np.arange(B * nblk, dtype=np.int32).reshape(B, nblk)
    seq_lens = np.full((B,), L, np.int32)
    return q, k, v, table, seq_lens


def contiguous_kv(k, v, b, g, L, nblk):
    """Logical rows of (b, g) from an identity layout, float64 [L, D]."""
    D = k.shape[-1]
    kk = widen(k[b * nblk:(b + 1) * nblk, g].reshape(-1, D)[:L])
    vv = widen(v[b * nblk:(b + 1) * nblk, g].reshape(-1, D)[:L])
    return kk, vv


def permute_pages(rng, k, v, table):
    """Relabel physical blocks by a random permutation pi: page i moves to
    slot pi[i] and every table entry follows it."""
    nb = k.shape[0]
    pi = rng.permutation(nb).astype(np.int32)
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[pi] = k
    v2[pi] = v
    t2 = np.where(table >= 0, pi[np.maximum(table, 0)], -1).astype(np.int32)
    return k2, v2, t2


def to_dev(a, device="cuda:0"):
    """numpy -> torch on the GPU; uint16 arrays become bfloat16 (same bits)."""
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_host(t):
    """torch (GPU) -> numpy; bfloat16 comes back as uint16 bit patterns."""
    import torch
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def out_as_f64(t):
    """GPU attention output widened to float64."""
    return widen(to_host(t))
