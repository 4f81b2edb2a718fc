"""Pins of the fp64 attention / KV-append oracle to facts fixed outside it:
the pages' worked statements, closed forms, a library routine (torch SDPA in
fp64, scipy softmax/logsumexp), structural invariances of a paged cache, and
the tiled algorithm agreeing with the full materialisation."""
import math

import numpy as np
import pytest
import scipy.special
import torch

from conftest import read_golden
from helpers import contiguous_kv, identity_layout, permute_pages, widen
from spec_verify_paged_gb300 import accounting as A
from spec_verify_paged_gb300 import workloads as W


def _run(oracle_mod, q, k, v, table, seq_lens, q_len, n_sink=0, window=0,
         scale=None, **kw):
    return oracle_mod.paged_attention(q, k, v, table, seq_lens, q_len, n_sink,
                                      window, scale, **kw)


def test_equal_scores_give_uniform_weights(oracle_mod):
    """StreamingLLM page, "The softmax problem": all-zero scores spread the
    mass evenly (0.25 each over four tokens).  One-hot V rows make the output
    equal to the attention weights themselves."""
    scores, probs = read_golden("softmax_equal_scores.txt")[0].split("|")
    n = len(scores.split())
    expect = np.array([float(x) for x in probs.split()])
    D = 16
    q = np.zeros((1, 1, 1, D), np.float32)          # every score is 0
    k = np.random.default_rng(0).standard_normal((1, 1, 16, D)).astype(np.float32)
    v = np.zeros((1, 1, 16, D), np.float32)
    for j in range(n):
        v[0, 0, j, j] = 1.0
    out, lse = _run(oracle_mod, q, k, v, np.zeros((1, 1), np.int32),
                    np.array([n], np.int32), 1)
    np.testing.assert_allclose(out[0, 0, 0, :n], expect, rtol=0, atol=1e-15)
    assert np.all(out[0, 0, 0, n:] == 0)
    assert lse[0, 0, 0] == pytest.approx(math.log(n), abs=1e-15)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_weights_match_scipy_softmax(oracle_mod, dtype):
    """With one-hot V rows the output row is softmax(scale * K q) itself:
    compare with scipy.special.softmax and logsumexp."""
    rng = np.random.default_rng(5)
    L, D = 45, 64
    q, k, _, table, sl = identity_layout(rng, 1, 1, D, L, dtype)
    v = np.zeros_like(k)
    one = np.float32(1.0) if dtype == "f32" else W.f32_to_bf16_bits(np.ones(1, np.float32))[0]
    for j in range(L):
        v[j // 16, 0, j % 16, j] = one
    scale = np.float32(0.3)
    out, lse = _run(oracle_mod, q, k, v, table, sl, 1, scale=scale)
    kk, _ = contiguous_kv(k, v, 0, 0, L, table.shape[1])
    s = float(scale) * (kk @ widen(q[0, 0, 0]))
    np.testing.assert_allclose(out[0, 0, 0, :L], scipy.special.softmax(s),
                               rtol=1e-12, atol=1e-15)
    assert lse[0, 0, 0] == pytest.approx(scipy.special.logsumexp(s), abs=1e-12)


@pytest.mark.parametrize("B,Hq,Hkv,D,L,dtype", [
    (2, 4, 4, 64, 37, "f32"),
    (1, 8, 2, 128, 100, "bf16"),
    (3, 6, 1, 64, 16, "bf16"),      # MQA
    (1, 4, 4, 64, 1, "f32"),        # a single cached row
])
def test_matches_torch_sdpa(oracle_mod, B, Hq, Hkv, D, L, dtype):
    """q_len 1, no window: plain softmax(q K^T * scale) V, which is exactly
    torch's scaled_dot_product_attention in float64 (GQA by repeating each
    kv head over its contiguous group of query heads)."""
    rng = np.random.default_rng(B * 100 + L)
    q, k, v, table, sl = identity_layout(rng, B, Hkv, D, L, dtype, Hq=Hq)
    scale = np.float32(1.0 / math.sqrt(D))
    out, lse = _run(oracle_mod, q, k, v, table, sl, 1, scale=scale)
    nblk = table.shape[1]
    G = Hq // Hkv
    for b in range(B):
        K = np.stack([contiguous_kv(k, v, b, g, L, nblk)[0] for g in range(Hkv)])
        V = np.stack([contiguous_kv(k, v, b, g, L, nblk)[1] for g in range(Hkv)])
        Kt = torch.from_numpy(K).repeat_interleave(G, dim=0)[None]
        Vt = torch.from_numpy(V).repeat_interleave(G, dim=0)[None]
        Qt = torch.from_numpy(widen(q[b, 0]))[None, :, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(
            Qt, Kt, Vt, scale=float(scale))[0, :, 0, :].numpy()
        np.testing.assert_allclose(out[b, 0], ref, rtol=0, atol=1e-12)
        s = float(scale) * np.einsum("hd,hjd->hj", widen(q[b, 0]),
                                     np.repeat(K, G, axis=0))
        np.testing.assert_allclose(lse[b, 0], scipy.special.logsumexp(s, axis=1),
                                   atol=1e-12)


@pytest.mark.parametrize("n_sink,window", [(0, 0), (2, 20), (0, 7)])
def test_verify_rows_equal_prefix_decodes(oracle_mod, n_sink, window):
    """"How speculative decoding doubles LLM speed", step 2: in the one
    verification pass each position attends to everything before it.  So
    query i of a q_len block equals a q_len-1 decode of the sequence cut
    right after it."""
    cfg = W.small_config(batch=3, num_q_heads=8, num_kv_heads=2, head_dim=64,
                         q_len=5, dtype="bf16", ctx_min=5, ctx_max=90, seed=3)
    wl = W.make_attention(cfg)
    out, lse = _run(oracle_mod, wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                    wl.seq_lens, 5, n_sink, window, wl.scale)
    for i in range(5):
        sl = wl.seq_lens - 5 + i + 1
        o1, l1 = _run(oracle_mod, np.ascontiguousarray(wl.q[:, i:i + 1]),
                      wl.k_cache, wl.v_cache, wl.block_table, sl, 1, n_sink,
                      window, wl.scale)
        assert np.array_equal(out[:, i], o1[:, 0])
        assert np.array_equal(lse[:, i], l1[:, 0])


def test_block_permutation_invariance(oracle_mod):
    """"KV cache & Flash Attention", section "PagedAttention": the page
    table only maps logical positions to physical blocks, so relabelling the
    blocks (moving the pages and the table entries together) changes
    nothing, bit for bit."""
    rng = np.random.default_rng(9)
    q, k, v, table, sl = identity_layout(rng, 3, 2, 64, 70, "bf16", Hq=4,
                                         q_len=3)
    sl = np.array([70, 33, 48], np.int32)
    ref = _run(oracle_mod, q, k, v, table, sl, 3, 1, 9, np.float32(0.125))
    for _ in range(3):
        k2, v2, t2 = permute_pages(rng, k, v, table)
        got = _run(oracle_mod, q, k2, v2, t2, sl, 3, 1, 9, np.float32(0.125))
        assert np.array_equal(ref[0], got[0]) and np.array_equal(ref[1], got[1])


def test_aliased_prefix_blocks(oracle_mod):
    """Sequences may share physical blocks (prefix sharing, "PagedAttention"
    section): a sequence reading two shared pages gives the same result as
    the same sequence with private copies of those pages."""
    rng = np.random.default_rng(4)
    q, k, v, table, sl = identity_layout(rng, 2, 2, 64, 64, "f32", Hq=2)
    shared = table.copy()
    shared[1, :2] = table[0, :2]                    # seq 1 aliases seq 0's pages
    private_k, private_v = k.copy(), v.copy()
    private_k[table[1, :2]] = k[table[0, :2]]       # copy them into seq 1's own
    private_v[table[1, :2]] = v[table[0, :2]]
    a = _run(oracle_mod, q, k, v, shared, sl, 1)
    b = _run(oracle_mod, q, private_k, private_v, table, sl, 1)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("tile,splits", [(1, 1), (4, 1), (16, 3), (5, 7), (64, 2)])
@pytest.mark.parametrize("n_sink,window", [(0, 0), (3, 25)])
def test_tiled_online_softmax_equals_full(oracle_mod, tile, splits, n_sink,
                                          window):
    """"KV cache & Flash Attention", "FlashAttention -- the tiling trick":
    the running (max, sum) makes the tiled result exact.  Split parts merged
    by log-sum-exp agree with full materialisation to fp64 rounding."""
    cfg = W.small_config(batch=2, num_q_heads=4, num_kv_heads=2, head_dim=64,
                         q_len=3, dtype="bf16", ctx_min=3, ctx_max=120, seed=7)
    wl = W.make_attention(cfg)
    full = _run(oracle_mod, wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                wl.seq_lens, 3, n_sink, window, wl.scale)
    tiled = _run(oracle_mod, wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                 wl.seq_lens, 3, n_sink, window, wl.scale,
                 tiled=(tile, splits))
    np.testing.assert_allclose(tiled[0], full[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(tiled[1], full[1], rtol=0, atol=1e-12)


GRID = [  # (seq_len, q_len, n_sink, window)
    (1, 1, 0, 0), (17, 1, 0, 0), (64, 4, 0, 0), (100, 1, 4, 20),
    (100, 5, 4, 20), (100, 3, 0, 1), (100, 2, 0, 7), (30, 1, 40, 5),
    (30, 1, 2, 64), (33, 8, 1, 3), (200, 1, 16, 16), (50, 2, 50, 1),
]


@pytest.mark.parametrize("L,q_len,n_sink,window", GRID)
def test_zero_query_gives_mean_and_log_count(oracle_mod, L, q_len, n_sink,
                                             window):
    """Q = 0 makes every score equal, so the weights are uniform over the
    visible set ("The softmax problem"): out is the mean of the visible V
    rows (one-hot V rows read the weights off directly) and lse = ln|V|.
    The count also pins the byte accounting's visible-set size."""
    D = 128
    rng = np.random.default_rng(L)
    nblk = -(-L // 16)
    k = rng.standard_normal((nblk, 1, 16, D)).astype(np.float32)
    v = np.zeros((nblk, 1, 16, D), np.float32)
    for j in range(min(L, D)):
        v[j // 16, 0, j % 16, j] = 1.0
    q = np.zeros((1, q_len, 1, D), np.float32)
    table = np.arange(nblk, dtype=np.int32)[None]
    out, lse = _run(oracle_mod, q, k, v, table, np.array([L], np.int32), q_len,
                    n_sink, window)
    for i in range(q_len):
        t = L - q_len + i
        n = A.visible_count(t, n_sink, window)
        assert lse[0, i, 0] == pytest.approx(math.log(n), abs=1e-13)
        w = out[0, i, 0, :min(L, D)]
        # the visible keys: the first n_sink and the last `window` up to t
        expect = np.zeros(min(L, D))
        for j in range(min(L, D)):
            if j <= t and (window == 0 or j < n_sink or j > t - window):
                expect[j] = 1.0 / n
        np.testing.assert_allclose(w, expect, rtol=0, atol=1e-15)
    # the union over the queries is what one call has to read
    union = A.union_visible_count(L, q_len, n_sink, window)
    seen = np.zeros(L, bool)
    for i in range(q_len):
        t = L - q_len + i
        for j in range(L):
            seen[j] |= j <= t and (window == 0 or j < n_sink or j > t - window)
    assert union == int(seen.sum())


def test_constant_values_give_that_constant(oracle_mod):
    """softmax weights sum to 1, so V rows all equal to c give exactly c."""
    rng = np.random.default_rng(2)
    q, k, v, table, sl = identity_layout(rng, 2, 2, 64, 50, "f32", Hq=4,
                                         q_len=2)
    c = rng.standard_normal(64).astype(np.float32)
    v[:] = c
    out, _ = _run(oracle_mod, q, k, v, table, sl, 2, 3, 10)
    np.testing.assert_allclose(out, np.broadcast_to(c.astype(np.float64),
                                                    out.shape), atol=1e-14)


def test_single_visible_key(oracle_mod):
    """window 1 and no sinks: each query sees only its own key, so out is
    that V row and lse its scaled score."""
    rng = np.random.default_rng(12)
    q, k, v, table, sl = identity_layout(rng, 1, 1, 64, 40, "bf16", q_len=3)
    out, lse = _run(oracle_mod, q, k, v, table, sl, 3, 0, 1, np.float32(0.5))
    kk, vv = contiguous_kv(k, v, 0, 0, 40, table.shape[1])
    for i in range(3):
        t = 40 - 3 + i
        np.testing.assert_array_equal(out[0, i, 0], vv[t])
        assert lse[0, i, 0] == pytest.approx(0.5 * kk[t] @ widen(q[0, i, 0]),
                                             abs=1e-12)


@pytest.mark.parametrize("n_sink,window", [(4, 37), (1, 16), (0, 9)])
def test_sink_window_equals_compacted_cache(oracle_mod, n_sink, window):
    """StreamingLLM page, "The StreamingLLM solution": keeping only the sink
    tokens plus the recent window and attending to all of them is what the
    sink+window mask computes in place.  Build the compacted cache (sinks,
    then the window rows, in order) and attend with no mask."""
    rng = np.random.default_rng(21)
    L, D = 200, 64
    q, k, v, table, sl = identity_layout(rng, 1, 2, D, L, "bf16", Hq=4)
    got = _run(oracle_mod, q, k, v, table, sl, 1, n_sink, window,
               np.float32(0.125))
    t = L - 1
    keep = list(range(n_sink)) + list(range(t - window + 1, t + 1))
    n = len(keep)
    nb = -(-n // 16)
    kc = np.zeros((nb, 2, 16, D), np.uint16)
    vc = np.zeros((nb, 2, 16, D), np.uint16)
    nblk = table.shape[1]
    for g in range(2):
        kf = k[:nblk, g].reshape(-1, D)
        vf = v[:nblk, g].reshape(-1, D)
        for r, j in enumerate(keep):
            kc[r // 16, g, r % 16] = kf[j]
            vc[r // 16, g, r % 16] = vf[j]
    ref = _run(oracle_mod, q, kc, vc, np.arange(nb, dtype=np.int32)[None],
               np.array([n], np.int32), 1, 0, 0, np.float32(0.125))
    np.testing.assert_allclose(got[0], ref[0], rtol=0, atol=1e-13)
    np.testing.assert_allclose(got[1], ref[1], rtol=0, atol=1e-13)


def test_stream_config_ring_cache(oracle_mod):
    """The full-size streaming workload: 1,000,000 positions, 4 sinks and a
    2044-key window held in a ring of pages.  Every query sees exactly
    4 + 2044 keys (lse of a zero query = ln 2048) and never touches a
    non-resident (NaN) row."""
    wl = W.make_attention(W.CONFIGS["stream-sink-window"])
    cfg = wl.cfg
    rows = np.array([0, 31, 5 * 32 + 7, 7 * 32 + 31], np.int64)
    out, lse = oracle_mod.paged_attention(
        wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.seq_lens, 1,
        cfg.n_sink, cfg.window, wl.scale, rows=rows)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    q0 = np.zeros_like(wl.q)
    _, lse0 = oracle_mod.paged_attention(
        q0, wl.k_cache, wl.v_cache, wl.block_table, wl.seq_lens, 1,
        cfg.n_sink, cfg.window, wl.scale, rows=rows)
    np.testing.assert_allclose(lse0, math.log(2048), atol=1e-12)


def test_poisoned_rows_are_never_read(oracle_mod):
    """Rows past seq_len hold NaN in the generated caches; a correct gather
    never touches them."""
    for q_len, n_sink, window in [(1, 0, 0), (4, 0, 0), (2, 3, 17)]:
        cfg = W.small_config(batch=4, q_len=q_len, ctx_min=q_len, ctx_max=70,
                             seed=30 + q_len)
        wl = W.make_attention(cfg)
        out, lse = oracle_mod.paged_attention(
            wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.seq_lens, q_len,
            n_sink, window, wl.scale)
        assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_bad_block_id_is_reported(oracle_mod):
    cfg = W.small_config(batch=1, ctx_min=40, ctx_max=40, seed=1)
    wl = W.make_attention(cfg)
    bt = wl.block_table.copy()
    bt[0, 1] = wl.num_blocks + 5
    with pytest.raises(ValueError):
        oracle_mod.paged_attention(wl.q, wl.k_cache, wl.v_cache, bt,
                                   wl.seq_lens, 1)


def test_kv_append_lands_at_the_new_positions(oracle_mod):
    """"KV cache & Flash Attention", "KV cache": each new token's K and V
    are stored at its position.  After the append, a window-1 query at each
    new position sees exactly the row that was appended there; no other
    cache element changes."""
    cfg = W.small_config(batch=3, num_q_heads=4, num_kv_heads=2, head_dim=64,
                         q_len=3, dtype="bf16", ctx_min=3, ctx_max=60, seed=8)
    wl = W.make_attention(cfg, n_new=3)
    kc, vc = oracle_mod.kv_append(wl.k_new, wl.v_new, wl.k_cache, wl.v_cache,
                                  wl.block_table, wl.seq_lens)
    changed = (kc != wl.k_cache).sum() + (vc != wl.v_cache).sum()
    assert changed == 2 * wl.k_new.size
    out, lse = oracle_mod.paged_attention(wl.q, kc, vc, wl.block_table,
                                          wl.seq_lens, 3, 0, 1, wl.scale)
    G = 2
    for b in range(3):
        for i in range(3):
            for h in range(4):
                np.testing.assert_array_equal(out[b, i, h],
                                              widen(wl.v_new[b, i, h // G]))
                s = float(wl.scale) * widen(wl.q[b, i, h]) @ widen(wl.k_new[b, i, h // G])
                assert lse[b, i, h] == pytest.approx(s, abs=1e-12)


def test_kv_bytes_formula_matches_pages():
    """KV bytes per token: 16,384 B / 512 KiB / 16 GiB (7B), 4,096 B / 10 GiB
    / 40 GiB (70B GQA), 80 GiB (MHA-64) from the lesson's "KV-cache math",
    and 524,288 B from the StreamingLLM page."""
    rows = read_golden("kv_bytes.txt")
    assert len(rows) == 8
    for row in rows:
        layers, heads, d, nbytes, tokens, expect = map(int, row.split()[:6])
        assert A.kv_bytes_per_token(layers, heads, d, nbytes) * tokens == expect
    per_token = A.kv_bytes_per_token(32, 32, 128, 2)
    for row in read_golden("kv_bytes_approx.txt"):
        tokens, approx, tol = (float(x) for x in row.split())
        assert abs(per_token * tokens - approx) <= tol * approx


def test_traffic_of_the_decode_workload():
    """decode-7b reads 16,384 B per cached token per call (one layer)."""
    sl = np.array([512, 4096, 1000])
    t = A.attention_traffic(sl, 1, 32, 32, 128, 2)
    assert t["kv_bytes"] == 16384 * int(sl.sum())
    assert t["flops"] == 4 * 32 * 128 * int(sl.sum())
    s = A.attention_traffic(np.array([1_000_000]), 1, 32, 32, 128, 2, 4, 2044)
    assert s["visible_rows"] == 2048
