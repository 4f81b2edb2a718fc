"""Seeded synthetic inputs shared by the CUDA path's tests/benchmark and the
CPU oracle.

This module holds no attention or acceptance arithmetic: it only draws random
numbers, rounds them once to the storage dtype, and lays them out (paged
caches, shuffled or ring-buffered block tables, logits, draft tokens,
uniforms).  Both sides read the very same bits.

Workloads (each named by what it is):
  tiny-decode         1 seq, 4/4 heads, D 64, context 256, q_len 1, fp32
  decode-7b           32 seqs, 32/32 heads (MHA), D 128, context U[512,4096],
                      q_len 1, bf16
  verify-gqa          16 seqs, 32/8 heads (GQA), D 128, context U[2048,8192]
                      including the 5 new rows, q_len 5 (causal draft), bf16;
                      acceptance on vocab 32000 with K = 4 drafts
  stream-sink-window  8 seqs, 32/32 heads, D 128, bf16, 4 sink + 2044 window
                      keys resident in a ring of pages after 1,000,000
                      streamed positions, sink keys scaled by 4
  long-context-128k   4 seqs, 64/8 heads, D 128, context 131072, q_len 1 or 4
All use 16-token pages ("KV cache & Flash Attention" lesson, section
"PagedAttention") and Q/K/V ~ N(0, 1); scale = 1/sqrt(D) held in fp32.

Layouts:
  q              [B, q_len, Hq, D]
  k/v cache      [num_blocks, Hkv, 16, D]   (one head's page is contiguous)
  block_table    [B, max_blocks_per_seq] int32, -1 = not resident
  seq_lens       [B] int32, logical length including the q_len new rows
bf16 tensors are carried as uint16 bit patterns (round-to-nearest-even from
fp32 draws).  Rows that a real cache would not hold valid data in (positions
at or past seq_len, evicted stream positions) are filled with NaN when
``poison=True`` so that a kernel touching them shows up.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

BLOCK_SIZE = 16
BF16_NAN = np.uint16(0x7FC0)


# --------------------------------------------------------------------------
# storage helpers (data preparation only)
# --------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bfloat16 (nearest, ties to even); returns uint16."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def _normals(rng: np.random.Generator, shape, dtype: str, chunk=1 << 24):
    """N(0,1) draws in fp32, stored as fp32 or as bf16 bits."""
    n = int(np.prod(shape))
    out = np.empty(n, np.float32 if dtype == "f32" else np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = rng.standard_normal(e - s, dtype=np.float32)
        out[s:e] = x if dtype == "f32" else f32_to_bf16_bits(x)
    return out.reshape(shape)


FP8_SCALE = 2.0 ** -5        # k_scale = v_scale of the FP8 workloads
FP8_NAN = np.uint8(0x7F)      # E4M3 NaN code


def _fp8_codes(x: np.ndarray, scale: float) -> np.ndarray:
    """E4M3 codes of fp32 values / scale, via torch's float8_e4m3fn cast
    (data preparation: the synthetic cache contents)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32) / np.float32(scale))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _kv_values(rng: np.random.Generator, shape, dtype: str):
    """Cache contents: N(0,1) draws stored as fp32, bf16 bits or, for
    "fp8", E4M3 codes of value / FP8_SCALE."""
    if dtype != "fp8":
        return _normals(rng, shape, dtype)
    n = int(np.prod(shape))
    out = np.empty(n, np.uint8)
    chunk = 1 << 24
    for s0 in range(0, n, chunk):
        e = min(n, s0 + chunk)
        out[s0:e] = _fp8_codes(rng.standard_normal(e - s0, dtype=np.float32),
                               FP8_SCALE)
    return out.reshape(shape)


def _nan_value(dtype: str):
    if dtype == "fp8":
        return FP8_NAN
    return np.float32(np.nan) if dtype == "f32" else BF16_NAN


def io_dtype(dtype: str) -> str:
    """Storage of q, out and new K/V rows: the cache's, except bf16 for an
    FP8 cache."""
    return "bf16" if dtype == "fp8" else dtype


# --------------------------------------------------------------------------
# attention workloads
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class AttnConfig:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    q_len: int
    dtype: str                 # cache: "f32", "bf16" or "fp8" (E4M3,
                               # q / out / new rows in bf16)
    ctx_min: int               # seq_len range (including the q_len new rows)
    ctx_max: int
    n_sink: int = 0
    window: int = 0
    ring: bool = False         # ring-buffered resident pages (streaming)
    sink_key_scale: float = 1.0
    seed: int = 0
    tree_depth: int = 0        # > 0: the q_len new rows are a complete
                               # binary draft tree of this depth


CONFIGS = {
    "tiny-decode": AttnConfig("tiny-decode", 1, 4, 4, 64, 1, "f32", 256, 256,
                              seed=1),
    "decode-7b": AttnConfig("decode-7b", 32, 32, 32, 128, 1, "bf16", 512,
                            4096, seed=2),
    "verify-gqa": AttnConfig("verify-gqa", 16, 32, 8, 128, 5, "bf16", 2048,
                             8192, seed=3),
    "stream-sink-window": AttnConfig("stream-sink-window", 8, 32, 32, 128, 1,
                                     "bf16", 1_000_000, 1_000_000, n_sink=4,
                                     window=2044, ring=True,
                                     sink_key_scale=4.0, seed=4),
    "long-context-128k": AttnConfig("long-context-128k", 4, 64, 8, 128, 1,
                                    "bf16", 131072, 131072, seed=5),
    # the 7B decode shape over an FP8 E4M3 cache (half the KV bytes)
    "decode-7b-fp8": AttnConfig("decode-7b-fp8", 32, 32, 32, 128, 1, "fp8",
                                512, 4096, seed=2),
    "long-context-128k-verify": AttnConfig("long-context-128k-verify", 4, 64,
                                           8, 128, 4, "bf16", 131072, 131072,
                                           seed=5),
    # SpecInfer-style draft tree: 2 candidates per depth, 3 levels, so
    # 1 + 2 + 4 + 8 = 15 new rows (the root and 14 draft nodes)
    "tree-verify": AttnConfig("tree-verify", 16, 32, 8, 128, 15, "bf16", 2048,
                              8192, seed=6, tree_depth=3),
}

ACCEPT_CONFIG = dict(name="verify-gqa-accept", batch=16, num_draft=4,
                     vocab=32000, target_std=2.0, noise_std=0.5, seed=3)
TREE_ACCEPT_CONFIG = dict(name="tree-verify-accept", batch=16, depth=3,
                          vocab=32000, target_std=2.0, noise_std=0.5, seed=6)


def binary_tree_parents(depth: int) -> np.ndarray:
    """Parents of a complete binary tree in breadth-first numbering: node 0
    is the root, node c >= 1 hangs below (c - 1) // 2; 2^(depth+1) - 1
    nodes."""
    n = (1 << (depth + 1)) - 1
    par = np.array([-1] + [(c - 1) // 2 for c in range(1, n)], np.int32)
    return par


def tree_mask_from_parents(parents: np.ndarray) -> np.ndarray:
    """Ancestor-or-self bit masks: bit k of entry i is set iff node k lies
    on the path from the root to node i (parents[..., c] < c).  Works on
    [N] or [B, N] arrays; returns uint32 of the same shape."""
    par = np.asarray(parents)
    mask = np.zeros(par.shape, np.uint32)
    for c in range(par.shape[-1]):
        own = np.uint32(1 << c)
        pc = par[..., c]
        if par.ndim == 1:
            mask[c] = own | (mask[pc] if pc >= 0 else np.uint32(0))
        else:
            up = np.where(pc >= 0, np.take_along_axis(
                mask, np.maximum(pc, 0)[:, None], axis=1)[:, 0], 0)
            mask[:, c] = own | up.astype(np.uint32)
    return mask


@dataclasses.dataclass
class AttnWorkload:
    cfg: AttnConfig
    q: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    block_table: np.ndarray
    seq_lens: np.ndarray
    scale: np.float32
    # rows to append before attending (kv_append inputs), may be None
    k_new: Optional[np.ndarray] = None
    v_new: Optional[np.ndarray] = None
    # [B, q_len] uint32 ancestor masks of a draft tree, or None (causal)
    tree_mask: Optional[np.ndarray] = None
    # FP8 caches: value = code * scale (1.0 otherwise)
    k_scale: float = 1.0
    v_scale: float = 1.0

    @property
    def q_len(self):
        return self.cfg.q_len

    @property
    def num_blocks(self):
        return self.k_cache.shape[0]

    @property
    def max_blocks_per_seq(self):
        return self.block_table.shape[1]


def _resident_positions(L: int, q_len: int, n_sink: int, window: int):
    """StreamingLLM cache policy (page "How StreamingLLM stabilizes
    million-token streams", section "The StreamingLLM solution"): the first
    n_sink positions plus the most recent window positions of the oldest new
    query, i.e. [0, n_sink) and [L - q_len - window + 1, L).  Returned as two
    half-open ranges."""
    lo = max(0, L - q_len - window + 1)
    return (0, min(n_sink, L)), (lo, L)


def make_attention(cfg: AttnConfig, seed: Optional[int] = None,
                   poison: bool = True, n_new: int = 0,
                   seq_lens: Optional[np.ndarray] = None,
                   spare_blocks: int = 0) -> AttnWorkload:
    """Build one attention workload.

    n_new > 0 additionally draws k_new/v_new [B, n_new, Hkv, D] for the last
    n_new positions of every sequence and poisons those cache rows, so the
    caller must kv_append them before attending.
    """
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    B, Hq, Hkv, D, ql = (cfg.batch, cfg.num_q_heads, cfg.num_kv_heads,
                         cfg.head_dim, cfg.q_len)
    if seq_lens is None:
        seq_lens = rng.integers(cfg.ctx_min, cfg.ctx_max + 1, size=B)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    assert seq_lens.shape == (B,) and (seq_lens >= ql).all()
    nblk = (seq_lens + BLOCK_SIZE - 1) // BLOCK_SIZE
    max_blocks = int(nblk.max()) if B else 0

    # which logical blocks hold data, and which positions are valid
    resident_blocks = []
    for b in range(B):
        L = int(seq_lens[b])
        if cfg.ring:
            (s0, s1), (w0, w1) = _resident_positions(L, ql, cfg.n_sink,
                                                     cfg.window)
            blocks = set(range(s0 // BLOCK_SIZE, (s1 + BLOCK_SIZE - 1) // BLOCK_SIZE))
            blocks |= set(range(w0 // BLOCK_SIZE, (w1 + BLOCK_SIZE - 1) // BLOCK_SIZE))
            resident_blocks.append(sorted(blocks))
        else:
            resident_blocks.append(list(range(int(nblk[b]))))

    # physical pages: one per resident logical block, except that a ring
    # layout folds the window blocks onto R reusable pages per sequence.
    phys_needed = []
    ring_sizes = []
    for b in range(B):
        if cfg.ring:
            n_sink_blocks = (min(cfg.n_sink, int(seq_lens[b])) + BLOCK_SIZE - 1) // BLOCK_SIZE
            R = -(-(cfg.window + ql - 1) // BLOCK_SIZE) + 1
            ring_sizes.append((n_sink_blocks, R))
            phys_needed.append(n_sink_blocks + R)
        else:
            phys_needed.append(len(resident_blocks[b]))
    num_blocks = int(sum(phys_needed)) + spare_blocks
    perm = rng.permutation(num_blocks).astype(np.int32)

    table = np.full((B, max(max_blocks, 1)), -1, np.int32)
    cursor = 0
    for b in range(B):
        ids = perm[cursor:cursor + phys_needed[b]]
        cursor += phys_needed[b]
        if cfg.ring:
            n_sink_blocks, R = ring_sizes[b]
            for lb in resident_blocks[b]:
                if lb < n_sink_blocks:
                    table[b, lb] = ids[lb]
                else:
                    table[b, lb] = ids[n_sink_blocks + (lb % R)]
        else:
            table[b, :len(ids)] = ids

    k_cache = _kv_values(rng, (num_blocks, Hkv, BLOCK_SIZE, D), cfg.dtype)
    v_cache = _kv_values(rng, (num_blocks, Hkv, BLOCK_SIZE, D), cfg.dtype)
    q = _normals(rng, (B, ql, Hq, D), io_dtype(cfg.dtype))

    if cfg.sink_key_scale != 1.0 and cfg.n_sink > 0 and cfg.dtype != "fp8":
        for b in range(B):
            for pos in range(min(cfg.n_sink, int(seq_lens[b]))):
                blk = table[b, pos // BLOCK_SIZE]
                row = k_cache[blk, :, pos % BLOCK_SIZE, :]
                f = (row.astype(np.float32) if cfg.dtype == "f32"
                     else bf16_bits_to_f32(row))
                f = f * np.float32(cfg.sink_key_scale)
                k_cache[blk, :, pos % BLOCK_SIZE, :] = (
                    f if cfg.dtype == "f32" else f32_to_bf16_bits(f))

    if poison:
        nan = _nan_value(cfg.dtype)
        for b in range(B):
            L = int(seq_lens[b])
            if cfg.ring:
                (s0, s1), (w0, w1) = _resident_positions(L, ql, cfg.n_sink,
                                                         cfg.window)
            # only the last page (and, for a ring, the resident pages) can
            # hold positions that carry no valid data
            cand = resident_blocks[b] if cfg.ring else resident_blocks[b][-1:]
            for lb in cand:
                blk = table[b, lb]
                for r in range(BLOCK_SIZE):
                    pos = lb * BLOCK_SIZE + r
                    valid = pos < L
                    if cfg.ring:
                        valid = (s0 <= pos < s1) or (w0 <= pos < w1)
                    if not valid:
                        k_cache[blk, :, r, :] = nan
                        v_cache[blk, :, r, :] = nan

    k_new = v_new = None
    if n_new > 0:
        k_new = _normals(rng, (B, n_new, Hkv, D), io_dtype(cfg.dtype))
        v_new = _normals(rng, (B, n_new, Hkv, D), io_dtype(cfg.dtype))
        nan = _nan_value(cfg.dtype)
        for b in range(B):
            L = int(seq_lens[b])
            for pos in range(L - n_new, L):
                blk = table[b, pos // BLOCK_SIZE]
                k_cache[blk, :, pos % BLOCK_SIZE, :] = nan
                v_cache[blk, :, pos % BLOCK_SIZE, :] = nan

    scale = np.float32(1.0 / math.sqrt(D))
    tree_mask = None
    if cfg.tree_depth > 0:
        par = binary_tree_parents(cfg.tree_depth)
        assert par.size == ql, "q_len must be the tree's node count"
        tree_mask = np.tile(tree_mask_from_parents(par), (B, 1))
    ks = FP8_SCALE if cfg.dtype == "fp8" else 1.0
    return AttnWorkload(cfg, q, k_cache, v_cache, table,
                        seq_lens.astype(np.int32), scale, k_new, v_new,
                        tree_mask, ks, ks)


def small_config(name="small", batch=3, num_q_heads=8, num_kv_heads=2,
                 head_dim=128, q_len=1, dtype="bf16", ctx_min=1, ctx_max=300,
                 n_sink=0, window=0, ring=False, sink_key_scale=1.0, seed=11):
    return AttnConfig(name, batch, num_q_heads, num_kv_heads, head_dim, q_len,
                      dtype, ctx_min, ctx_max, n_sink, window, ring,
                      sink_key_scale, seed)


# --------------------------------------------------------------------------
# acceptance workloads
# --------------------------------------------------------------------------

@dataclasses.dataclass
class AcceptWorkload:
    target_logits: np.ndarray   # [B, K+1, V] fp32
    draft_logits: np.ndarray    # [B, K, V] fp32
    draft_tokens: np.ndarray    # [B, K] int32, drawn from softmax(draft)
    uniforms: np.ndarray        # [B, K+1] fp32 in [0, 1)


def uniforms01(rng: np.random.Generator, shape) -> np.ndarray:
    """fp32 uniforms on the grid k * 2^-24, k in [0, 2^24): exact in fp32."""
    return (rng.integers(0, 1 << 24, size=shape).astype(np.float64)
            * 2.0 ** -24).astype(np.float32)


def make_accept(batch=16, num_draft=4, vocab=32000, target_std=2.0,
                noise_std=0.5, seed=3, **_unused) -> AcceptWorkload:
    """Target logits ~ N(0, target_std^2); draft logits = target (first K
    rows) + N(0, noise_std^2); draft tokens drawn from the draft softmax by
    the Gumbel-max trick (argmax of logits + Gumbel noise); uniforms in
    [0, 1)."""
    rng = np.random.default_rng(seed)
    B, K, V = batch, num_draft, vocab
    target = (rng.standard_normal((B, K + 1, V), dtype=np.float32)
              * np.float32(target_std))
    draft = (target[:, :K, :] + rng.standard_normal((B, K, V), dtype=np.float32)
             * np.float32(noise_std)).astype(np.float32)
    gumbel = rng.gumbel(size=(B, K, V))
    tokens = np.argmax(draft.astype(np.float64) + gumbel, axis=-1).astype(np.int32)
    u = uniforms01(rng, (B, K + 1))
    return AcceptWorkload(target.astype(np.float32), draft, tokens, u)


@dataclasses.dataclass
class TreeAcceptWorkload:
    target_logits: np.ndarray   # [B, N, V] fp32: row i = target after node i
    draft_logits: np.ndarray    # [B, N, V] fp32: row i = draft after node i
    parents: np.ndarray         # [B, N] int32, parents[:, 0] = -1
    node_tokens: np.ndarray     # [B, N] int32 (entry 0 unused: -1)
    uniforms: np.ndarray        # [B, N] fp32 in [0, 1)


def make_tree_accept(batch=16, depth=3, vocab=32000, target_std=2.0,
                     noise_std=0.5, seed=6, parents=None,
                     **_unused) -> TreeAcceptWorkload:
    """A draft tree per sequence (complete binary of `depth` levels unless
    `parents` [N] is given).  Target logits ~ N(0, target_std^2) per node;
    draft logits = target + N(0, noise_std^2); the children of node i are
    drawn independently from softmax(draft row i) by the Gumbel-max trick
    (the draft model sampling several continuations); uniforms in [0, 1)."""
    rng = np.random.default_rng(seed)
    par = binary_tree_parents(depth) if parents is None else np.asarray(
        parents, np.int32)
    B, N, V = batch, par.size, vocab
    target = (rng.standard_normal((B, N, V), dtype=np.float32)
              * np.float32(target_std))
    draft = (target + rng.standard_normal((B, N, V), dtype=np.float32)
             * np.float32(noise_std)).astype(np.float32)
    tokens = np.full((B, N), -1, np.int32)
    for c in range(1, N):
        g = rng.gumbel(size=(B, V))
        tokens[:, c] = np.argmax(draft[:, par[c], :].astype(np.float64) + g,
                                 axis=-1)
    u = uniforms01(rng, (B, N))
    return TreeAcceptWorkload(target.astype(np.float32), draft,
                              np.tile(par, (B, 1)).astype(np.int32), tokens, u)
