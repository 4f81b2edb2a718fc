"""GPU draft-tree attention vs the fp64 oracle, element by element.

Same tolerances as the causal block: max |out - oracle| <= 2e-2 for bf16
KV, 1e-5 for fp32 KV; |lse - oracle| <= 1e-3."""
import numpy as np
import pytest

from helpers import out_as_f64, to_dev
from spec_verify_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-5}
LSE_TOL = 1e-3
PATHS = {"auto": 0, "cuda_cores": 1, "tensor_cores": 2, "tcgen05": 3}


@pytest.fixture(scope="module")
def svp():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import spec_verify_paged_gb300 as m
    return m


def _random_parents(rng, n):
    return np.array([-1] + [int(rng.integers(0, c)) for c in range(1, n)],
                    np.int32)


def _masks(kind, B, n, seed):
    rng = np.random.default_rng(seed)
    if kind == "binary":
        depth = {3: 1, 7: 2, 15: 3}[n]
        par = np.tile(W.binary_tree_parents(depth), (B, 1))
    elif kind == "chain":
        par = np.tile(np.arange(-1, n - 1, dtype=np.int32), (B, 1))
    elif kind == "star":
        par = np.tile(np.array([-1] + [0] * (n - 1), np.int32), (B, 1))
    else:  # a different random tree per sequence
        par = np.stack([_random_parents(rng, n) for _ in range(B)])
    return W.tree_mask_from_parents(par)


def _run_gpu(svp, wl, mask, kernel_path=0, split_pages=0):
    import torch
    kc, vc = to_dev(wl.k_cache), to_dev(wl.v_cache)
    bt, sl = to_dev(wl.block_table), to_dev(wl.seq_lens)
    if wl.k_new is not None:
        svp.kv_append(to_dev(wl.k_new), to_dev(wl.v_new), kc, vc, bt, sl)
    tm = to_dev(mask.view(np.int32))
    out, lse = svp.paged_tree_attention(to_dev(wl.q), kc, vc, bt, sl, tm,
                                        scale=float(wl.scale),
                                        kernel_path=kernel_path,
                                        split_pages=split_pages)
    torch.cuda.synchronize()
    assert svp.read_device_status() == 0
    return out_as_f64(out), lse.cpu().numpy().astype(np.float64)


def _oracle(oracle_mod, wl, mask, rows=None):
    kc, vc = wl.k_cache, wl.v_cache
    if wl.k_new is not None:
        kc, vc = oracle_mod.kv_append(wl.k_new, wl.v_new, kc, vc,
                                      wl.block_table, wl.seq_lens)
    return oracle_mod.paged_tree_attention(wl.q, kc, vc, wl.block_table,
                                           wl.seq_lens, wl.q_len, mask,
                                           wl.scale, rows=rows)


def _compare(dtype, got, ref, rows=None):
    out, lse = got
    o_ref, l_ref = ref
    if rows is not None:
        D = out.shape[-1]
        out = out.reshape(-1, D)[rows]
        lse = lse.reshape(-1)[rows]
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    err = np.abs(out - o_ref).max()
    lerr = np.abs(lse - l_ref).max()
    assert err <= TOL[dtype], f"max |out err| {err}"
    assert lerr <= LSE_TOL, f"max |lse err| {lerr}"


CASES = [
    # (tree, q_len, dtype, D, Hq, Hkv, ctx_min, ctx_max, split_pages)
    ("binary", 15, "bf16", 128, 32, 8, 15, 600, 0),   # the tree-verify shape
    ("binary", 7, "bf16", 128, 8, 2, 7, 300, 2),
    ("binary", 3, "f32", 64, 4, 4, 3, 200, 0),
    ("random", 16, "bf16", 128, 8, 8, 16, 400, 3),
    ("random", 9, "bf16", 64, 8, 2, 9, 250, 1),
    ("star", 6, "bf16", 128, 16, 4, 6, 180, 0),
    ("random", 12, "f32", 128, 4, 2, 12, 130, 2),
    ("binary", 15, "bf16", 128, 32, 8, 15, 15, 0),    # nothing but the tree
]


def _unsupported(path, dtype, D):
    if path == "tensor_cores":
        return dtype == "f32"
    if path == "tcgen05":
        return dtype == "f32" or D != 128
    return False


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_tree_parity(svp, oracle_mod, case, path):
    kind, n, dtype, D, Hq, Hkv, lo, hi, sp = case
    if _unsupported(path, dtype, D):
        pytest.skip("path does not take this dtype / head_dim")
    cfg = W.small_config(batch=5, num_q_heads=Hq, num_kv_heads=Hkv,
                         head_dim=D, q_len=n, dtype=dtype, ctx_min=lo,
                         ctx_max=hi, seed=300 + n + D + Hq)
    wl = W.make_attention(cfg, n_new=n)
    mask = _masks(kind, 5, n, seed=n)
    got = _run_gpu(svp, wl, mask, kernel_path=PATHS[path], split_pages=sp)
    _compare(dtype, got, _oracle(oracle_mod, wl, mask))


@pytest.mark.parametrize("path", [1, 2, 3])
def test_chain_tree_equals_causal_block(svp, path):
    """A chain mask is the causal verify block: the tree call returns
    exactly what the causal call returns on the same kernel path."""
    import torch
    cfg = W.small_config(batch=4, num_q_heads=16, num_kv_heads=4,
                         head_dim=128, q_len=5, dtype="bf16", ctx_min=5,
                         ctx_max=500, seed=41)
    wl = W.make_attention(cfg)
    mask = _masks("chain", 4, 5, 0)
    got = _run_gpu(svp, wl, mask, kernel_path=path)
    kc, vc = to_dev(wl.k_cache), to_dev(wl.v_cache)
    out, lse = svp.paged_decode_attention(
        to_dev(wl.q), kc, vc, to_dev(wl.block_table), to_dev(wl.seq_lens),
        q_len=5, scale=float(wl.scale), kernel_path=path)
    torch.cuda.synchronize()
    assert np.array_equal(got[0], out_as_f64(out))
    assert np.array_equal(got[1], lse.cpu().numpy().astype(np.float64))


def test_tree_verify_config_sampled(svp, oracle_mod):
    """The tree-verify workload at full size (16 sequences, 32/8 heads,
    15-node binary tree, contexts 2k-8k), automatic path as benchmarked,
    compared on sampled rows including every node of the first and last
    sequence."""
    cfg = W.CONFIGS["tree-verify"]
    wl = W.make_attention(cfg, n_new=cfg.q_len)
    got = _run_gpu(svp, wl, wl.tree_mask)
    rng = np.random.default_rng(5)
    per = cfg.q_len * cfg.num_q_heads
    rows = np.unique(np.concatenate([
        rng.choice(cfg.batch * per, 64, replace=False),
        np.arange(0, per, cfg.num_q_heads),
        (cfg.batch - 1) * per + np.arange(0, per, cfg.num_q_heads) + 31,
    ])).astype(np.int64)
    ref = _oracle(oracle_mod, wl, wl.tree_mask, rows=rows)
    _compare(cfg.dtype, got, ref, rows=rows)

