"""Algorithmic byte and FLOP accounting for the decode/verify attention
metric (KV-read GB/s and query-tokens/s).

KV bytes per token follow the formula of the lesson "KV cache & Flash
Attention" (section "KV-cache math") and of the StreamingLLM page (section
"The KV cache memory bottleneck"): 2 (K and V) x layers x kv_heads x head_dim
x bytes per element.  A call reads each visible cached row of a sequence
once for all of its q_len queries and all query heads of a GQA group, so the
algorithmic KV bytes of one call are, per sequence,
2 x Hkv x D x bytes x |union over queries of the visible set|.
"""
from __future__ import annotations

import numpy as np


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int,
                       bytes_per_elem: int) -> int:
    """2 * layers * kv_heads * head_dim * bytes_per_elem (K and V)."""
    return 2 * layers * kv_heads * head_dim * bytes_per_elem


def visible_count(t: int, n_sink: int, window: int) -> int:
    """Number of keys visible to a query at absolute position t: keys
    0..t (causal), restricted to the first n_sink plus the last `window`
    (own key included) when window > 0."""
    if t < 0:
        return 0
    if window == 0:
        return t + 1
    sinks = min(n_sink, t + 1)
    lo = max(0, t - window + 1)          # first key of the window
    recent = t + 1 - lo
    overlap = max(0, min(n_sink, t + 1) - lo)
    return sinks + recent - overlap


def union_visible_count(seq_len: int, q_len: int, n_sink: int,
                        window: int) -> int:
    """Rows read once per (sequence, kv head): the union of the visible sets
    of the q_len queries at positions seq_len-q_len .. seq_len-1."""
    if window == 0:
        return seq_len
    t0 = seq_len - q_len
    lo = max(0, t0 - window + 1)
    recent = seq_len - lo
    overlap = max(0, min(n_sink, seq_len) - lo)
    return min(n_sink, seq_len) + recent - overlap


def attention_traffic(seq_lens, q_len: int, num_q_heads: int,
                      num_kv_heads: int, head_dim: int, elem_bytes: int,
                      n_sink: int = 0, window: int = 0) -> dict:
    """Algorithmic bytes and FLOPs of one paged_decode_attention call (one
    layer).  kv_bytes counts every visible K and V row once; io_bytes adds
    q, out, lse and the touched block-table entries; flops = 4 * Hq * D *
    sum over queries of |visible set| (QK^T and PV, 2 flops per MAC)."""
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    rows = 0
    vis = 0
    for L in seq_lens.tolist():
        rows += union_visible_count(L, q_len, n_sink, window)
        for i in range(q_len):
            vis += visible_count(L - q_len + i, n_sink, window)
    kv = 2 * num_kv_heads * head_dim * elem_bytes * rows
    B = len(seq_lens)
    q_bytes = B * q_len * num_q_heads * head_dim * elem_bytes
    lse_bytes = B * q_len * num_q_heads * 4
    table_bytes = 4 * sum(-(-int(union_visible_count(L, q_len, n_sink, window)) // 16) + 1
                          for L in seq_lens.tolist())
    return {
        "kv_bytes": int(kv),
        "io_bytes": int(kv + 2 * q_bytes + lse_bytes + table_bytes),
        "flops": int(4 * num_q_heads * head_dim * vis),
        "query_tokens": int(B * q_len),
        "visible_rows": int(rows),
    }


def accept_traffic(batch: int, num_draft: int, vocab: int) -> dict:
    """One spec_accept call reads every target and draft logit once."""
    logits = batch * (2 * num_draft + 1) * vocab * 4
    return {"logit_bytes": int(logits),
            "io_bytes": int(logits + batch * (num_draft * 4 + (num_draft + 1) * 8 + 4))}
