"""Pins of the FP8 (E4M3) KV-cache oracle.

The KV-cache lesson ("KV cache & Flash Attention", section "Practical use")
serves with an fp8 KV cache and the StreamingLLM page ("The KV cache memory
bottleneck") lists KV quantisation; neither fixes the format, so the build
reads it as OCP E4M3 codes times a per-cache scale.  Pins: the oracle's
decoding and rounding equal torch's float8_e4m3fn conversion (a library
routine), saturation follows the format's largest finite value, and
attention over an FP8 cache equals torch SDPA (fp64) over the dequantised
values."""
import math

import numpy as np
import pytest
import torch

from helpers import contiguous_kv, identity_layout, widen
from spec_verify_paged_gb300 import workloads as W


def test_decode_matches_torch_float8():
    import oracle
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9   # max, min subnormal


def test_encode_matches_torch_float8_including_ties():
    import oracle
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(200_000).astype(np.float32) * 40,
        rng.standard_normal(20_000).astype(np.float32) * 1e-2,   # subnormals
    ])
    # exact midpoints between neighbouring codes: ties to the even code
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids])
    x = x[np.abs(x) <= 448]
    mine = oracle.e4m3_encode(x, 1.0)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)
    assert np.all(mine[-2 * mids.size:-mids.size] & 1 == 0)  # ties went even


def test_encode_saturates_and_scales():
    import oracle
    big = np.array([448.0, 449.0, 464.0, 1e6, -500.0], np.float32)
    assert list(oracle.e4m3_encode(big, 1.0)) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]
    # value / scale with a power-of-two scale is the same code as value
    x = np.array([0.75, -3.0, 13.0], np.float32)
    assert np.array_equal(oracle.e4m3_encode(x * 2 ** -5, 2 ** -5),
                          oracle.e4m3_encode(x, 1.0))


@pytest.mark.parametrize("Hq,Hkv,L", [(4, 4, 37), (8, 2, 100)])
def test_fp8_attention_matches_sdpa_on_dequantised_cache(Hq, Hkv, L):
    import oracle
    rng = np.random.default_rng(Hq + L)
    B, D = 2, 64
    q, k, v, table, sl = identity_layout(rng, B, Hkv, D, L, "bf16", Hq=Hq)
    ks, vs = 2.0 ** -5, 2.0 ** -4
    kf = W._fp8_codes(widen(k).astype(np.float32), ks)
    vf = W._fp8_codes(widen(v).astype(np.float32), vs)
    scale = np.float32(1 / math.sqrt(D))
    out, lse = oracle.paged_attention_fp8(q, kf, vf, ks, vs, table, sl, 1,
                                          scale=scale)
    deq_k = torch.from_numpy(kf).view(torch.float8_e4m3fn).to(torch.float64) * ks
    deq_v = torch.from_numpy(vf).view(torch.float8_e4m3fn).to(torch.float64) * vs
    nblk = table.shape[1]
    G = Hq // Hkv
    for b in range(B):
        K = torch.stack([deq_k[b * nblk:(b + 1) * nblk, g].reshape(-1, D)[:L]
                         for g in range(Hkv)])
        V = torch.stack([deq_v[b * nblk:(b + 1) * nblk, g].reshape(-1, D)[:L]
                         for g in range(Hkv)])
        Qt = torch.from_numpy(widen(q[b, 0]))[None, :, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(
            Qt, K.repeat_interleave(G, 0)[None], V.repeat_interleave(G, 0)[None],
            scale=float(scale))[0, :, 0, :].numpy()
        np.testing.assert_allclose(out[b, 0], ref, rtol=0, atol=1e-12)


def test_fp8_append_stores_torch_codes_and_reads_back():
    """Appended rows are stored as the E4M3 codes of bf16 value / scale; a
    window-1 query at each new position reads exactly that row back."""
    import oracle
    cfg = W.small_config(batch=3, num_q_heads=4, num_kv_heads=2, head_dim=64,
                         q_len=3, dtype="fp8", ctx_min=3, ctx_max=50, seed=9)
    wl = W.make_attention(cfg, n_new=3)
    kc, vc = oracle.kv_append_fp8(wl.k_new, wl.v_new, wl.k_cache, wl.v_cache,
                                  wl.k_scale, wl.v_scale, wl.block_table,
                                  wl.seq_lens)
    for b in range(3):
        L = int(wl.seq_lens[b])
        for k in range(3):
            pos = L - 3 + k
            blk = wl.block_table[b, pos // 16]
            want = W._fp8_codes(widen(wl.k_new[b, k]).astype(np.float32),
                                wl.k_scale)
            assert np.array_equal(kc[blk, :, pos % 16], want)
    out, _ = oracle.paged_attention_fp8(wl.q, kc, vc, wl.k_scale, wl.v_scale,
                                        wl.block_table, wl.seq_lens, 3,
                                        window=1, scale=wl.scale)
    for b in range(3):
        for k in range(3):
            row = oracle.e4m3_decode(W._fp8_codes(
                widen(wl.v_new[b, k]).astype(np.float32), wl.v_scale)) * wl.v_scale
            for h in range(4):
                np.testing.assert_allclose(out[b, k, h], row[h // 2], atol=1e-12)
