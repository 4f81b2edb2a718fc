"""GPU attention over an FP8 E4M3 KV cache, and the quantising append, vs
the fp64 oracle.  The append's codes must be identical (byte work); the
attention has the bf16 tolerance (max |out - oracle| <= 2e-2, |lse| <= 1e-3):
both sides read the same stored codes, so the quantisation error is common
to both."""
import numpy as np
import pytest

from helpers import out_as_f64, to_dev
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


def _run(svp, wl, n_sink=0, window=0, kernel_path=0, split_pages=0):
    import torch
    kc, vc = to_dev(wl.k_cache), to_dev(wl.v_cache)
    bt, sl = to_dev(wl.block_table), to_dev(wl.seq_lens)
    if wl.k_new is not None:
        svp.kv_append(to_dev(wl.k_new), to_dev(wl.v_new), kc, vc, bt, sl,
                      k_scale=wl.k_scale, v_scale=wl.v_scale)
    out, lse = svp.paged_decode_attention(
        to_dev(wl.q), kc, vc, bt, sl, q_len=wl.q_len, n_sink=n_sink,
        window=window, scale=float(wl.scale), k_scale=wl.k_scale,
        v_scale=wl.v_scale, kernel_path=kernel_path, split_pages=split_pages)
    torch.cuda.synchronize()
    assert svp.read_device_status() == 0
    return (out_as_f64(out), lse.cpu().numpy().astype(np.float64),
            kc.cpu().numpy(), vc.cpu().numpy())


def _oracle(oracle_mod, wl, n_sink=0, window=0, rows=None):
    kc, vc = oracle_mod.kv_append_fp8(wl.k_new, wl.v_new, wl.k_cache,
                                      wl.v_cache, wl.k_scale, wl.v_scale,
                                      wl.block_table, wl.seq_lens)
    out, lse = oracle_mod.paged_attention_fp8(
        wl.q, kc, vc, wl.k_scale, wl.v_scale, wl.block_table, wl.seq_lens,
        wl.q_len, n_sink, window, wl.scale, rows=rows)
    return out, lse, kc, vc


def _compare(got, ref, rows=None):
    out, lse = got[0], got[1]
    if rows is not None:
        D = out.shape[-1]
        out = out.reshape(-1, D)[rows]
        lse = lse.reshape(-1)[rows]
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    assert np.abs(out - ref[0]).max() <= 2e-2
    assert np.abs(lse - ref[1]).max() <= 1e-3


CASES = [
    # (D, Hq, Hkv, q_len, ctx_min, ctx_max, n_sink, window, split_pages)
    (128, 8, 8, 1, 1, 600, 0, 0, 0),
    (64, 4, 4, 1, 1, 300, 0, 0, 2),
    (128, 16, 4, 5, 5, 700, 0, 0, 0),
    (128, 8, 2, 8, 8, 260, 0, 0, 3),
    (64, 8, 1, 3, 3, 200, 0, 0, 1),
    (128, 4, 4, 1, 1, 500, 4, 37, 0),
    (128, 8, 2, 4, 4, 500, 4, 37, 1),
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_fp8_parity(svp, oracle_mod, case):
    D, Hq, Hkv, q_len, lo, hi, n_sink, window, sp = case
    cfg = W.small_config(batch=5, num_q_heads=Hq, num_kv_heads=Hkv,
                         head_dim=D, q_len=q_len, dtype="fp8", ctx_min=lo,
                         ctx_max=hi, seed=500 + D + q_len + Hq)
    wl = W.make_attention(cfg, n_new=q_len)
    got = _run(svp, wl, n_sink, window, split_pages=sp)
    ref = _oracle(oracle_mod, wl, n_sink, window)
    # the append's codes are byte-identical
    assert np.array_equal(got[2], ref[2]) and np.array_equal(got[3], ref[3])
    _compare(got, ref)


def test_forced_tensor_paths_refuse_fp8(svp):
    cfg = W.small_config(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128,
                         q_len=4, dtype="fp8", ctx_min=4, ctx_max=60, seed=3)
    wl = W.make_attention(cfg, n_new=4)
    for path in (2, 3):
        with pytest.raises(svp.SvpError) as e:
            _run(svp, wl, kernel_path=path)
        assert e.value.status == -2


def test_decode_7b_fp8_sampled(svp, oracle_mod):
    """The decode-7b shape over an FP8 cache, at full size, on sampled rows."""
    cfg = W.CONFIGS["decode-7b-fp8"]
    wl = W.make_attention(cfg, n_new=1)
    got = _run(svp, wl)
    rng = np.random.default_rng(2)
    per = cfg.num_q_heads
    rows = np.unique(np.concatenate([rng.choice(cfg.batch * per, 96, replace=False),
                                     [0, cfg.batch * per - 1]])).astype(np.int64)
    ref = _oracle(oracle_mod, wl, rows=rows)
    _compare(got, ref, rows=rows)


def test_fp8_cache_with_a_tree_mask(svp, oracle_mod):
    """The draft-tree mask over an FP8 cache (CUDA-core path), against the
    fp32 tree oracle run over the dequantised cache: every E4M3 value times
    the power-of-two scale is exact in fp32, so both read the same keys and
    values (the poisoned rows past each sequence are never visible)."""
    import torch
    depth = 2
    n = (1 << (depth + 1)) - 1
    cfg = W.small_config(batch=3, num_q_heads=8, num_kv_heads=2, head_dim=128,
                         q_len=n, dtype="fp8", ctx_min=n + 1, ctx_max=300,
                         seed=77)
    wl = W.make_attention(cfg, n_new=n)
    par = W.binary_tree_parents(depth)
    mask = np.tile(W.tree_mask_from_parents(par), (3, 1))
    kc, vc = to_dev(wl.k_cache), to_dev(wl.v_cache)
    bt, sl = to_dev(wl.block_table), to_dev(wl.seq_lens)
    svp.kv_append(to_dev(wl.k_new), to_dev(wl.v_new), kc, vc, bt, sl,
                  k_scale=wl.k_scale, v_scale=wl.v_scale)
    out, lse = svp.paged_tree_attention(
        to_dev(wl.q), kc, vc, bt, sl, to_dev(mask.view(np.int32)),
        scale=float(wl.scale), k_scale=wl.k_scale, v_scale=wl.v_scale)
    torch.cuda.synchronize()
    assert svp.read_device_status() == 0
    got_o, got_l = out_as_f64(out), lse.cpu().numpy().astype(np.float64)
    # reference: dequantise the appended cache into fp32 and run the fp32
    # tree oracle over it (fp32 holds every E4M3 value times a power of two)
    kq, vq = oracle_mod.kv_append_fp8(wl.k_new, wl.v_new, wl.k_cache,
                                      wl.v_cache, wl.k_scale, wl.v_scale,
                                      wl.block_table, wl.seq_lens)
    kf = (oracle_mod.e4m3_decode(kq) * wl.k_scale).astype(np.float32)
    vf = (oracle_mod.e4m3_decode(vq) * wl.v_scale).astype(np.float32)
    kf = np.nan_to_num(kf, nan=0.0)
    vf = np.nan_to_num(vf, nan=0.0)
    qf = W.bf16_bits_to_f32(wl.q)
    ref_o, ref_l = oracle_mod.paged_tree_attention(qf, kf, vf, wl.block_table,
                                                   wl.seq_lens, n, mask,
                                                   wl.scale)
    assert np.abs(got_o - ref_o).max() <= 2e-2
    assert np.abs(got_l - ref_l).max() <= 1e-3
