"""GPU paged decode/verify attention vs the fp64 oracle, element by element.

Tolerances (stated by the workload definition): max |out - oracle| <= 2e-2
for bf16 KV and 1e-5 for fp32 KV; |lse - oracle| <= 1e-3."""
import numpy as np
import pytest

from helpers import out_as_f64, to_dev
from spec_verify_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-5}
LSE_TOL = 1e-3


@pytest.fixture(scope="module")
def svp():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import spec_verify_paged_gb300 as m
    return m


def _run_gpu(svp, wl, n_sink, window, split_pages=0, append=True,
             kernel_path=0):
    import torch
    kc, vc = to_dev(wl.k_cache), to_dev(wl.v_cache)
    bt, sl = to_dev(wl.block_table), to_dev(wl.seq_lens)
    if append and wl.k_new is not None:
        svp.kv_append(to_dev(wl.k_new), to_dev(wl.v_new), kc, vc, bt, sl)
    out, lse = svp.paged_decode_attention(
        to_dev(wl.q), kc, vc, bt, sl, q_len=wl.q_len, n_sink=n_sink,
        window=window, scale=float(wl.scale), split_pages=split_pages,
        kernel_path=kernel_path)
    torch.cuda.synchronize()
    assert svp.read_device_status() == 0
    return out_as_f64(out), lse.cpu().numpy().astype(np.float64)


def _compare(wl, got, ref, rows=None):
    out, lse = got
    o_ref, l_ref = ref
    if rows is not None:
        D = out.shape[-1]
        out = out.reshape(-1, D)[rows]
        lse = lse.reshape(-1)[rows]
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    err = np.abs(out - o_ref).max()
    lerr = np.abs(lse - l_ref).max()
    assert err <= TOL[wl.cfg.dtype], f"max |out err| {err}"
    assert lerr <= LSE_TOL, f"max |lse err| {lerr}"
    return err, lerr


def _oracle(oracle_mod, wl, n_sink, window, rows=None):
    kc, vc = wl.k_cache, wl.v_cache
    if wl.k_new is not None:
        kc, vc = oracle_mod.kv_append(wl.k_new, wl.v_new, kc, vc,
                                      wl.block_table, wl.seq_lens)
    return oracle_mod.paged_attention(wl.q, kc, vc, wl.block_table,
                                      wl.seq_lens, wl.q_len, n_sink, window,
                                      wl.scale, rows=rows)


SWEEP = [
    # (dtype, D, Hq, Hkv, q_len, ctx_min, ctx_max, n_sink, window, split_pages)
    ("f32", 64, 4, 4, 1, 1, 300, 0, 0, 0),
    ("f32", 128, 4, 2, 3, 3, 170, 0, 0, 2),
    ("bf16", 64, 8, 1, 1, 1, 90, 0, 0, 1),       # MQA, one page per split
    ("bf16", 128, 8, 8, 1, 1, 520, 0, 0, 0),
    ("bf16", 128, 16, 4, 2, 2, 400, 0, 0, 3),
    ("bf16", 128, 32, 8, 5, 5, 700, 0, 0, 0),     # verify shape: 20 rows
    ("bf16", 128, 8, 2, 8, 8, 260, 0, 0, 2),      # 32 rows, 4 row groups
    ("bf16", 64, 4, 1, 16, 16, 150, 0, 0, 0),     # q_len 16
    ("bf16", 128, 4, 4, 1, 1, 500, 4, 37, 0),     # sinks + window
    ("bf16", 128, 8, 2, 4, 4, 500, 4, 37, 1),
    ("bf16", 128, 4, 4, 1, 1, 300, 0, 16, 0),     # pure sliding window
    ("bf16", 128, 4, 4, 3, 3, 300, 20, 5, 2),     # sinks span 2 pages
    ("f32", 64, 2, 2, 2, 2, 200, 0, 1, 0),        # window 1: own key only
    ("bf16", 128, 8, 8, 1, 1, 64, 100, 8, 0),     # n_sink beyond the length
    ("bf16", 128, 12, 4, 3, 3, 300, 0, 0, 0),     # GQA group 3: Q row by row
    ("bf16", 128, 128, 1, 1, 1, 200, 0, 0, 0),    # group 128: two 64-row units
]


PATHS = {"auto": 0, "cuda_cores": 1, "tensor_cores": 2, "tcgen05": 3}


def _unsupported(path, dtype, D):
    """Forced tensor paths refuse data they cannot take."""
    if path == "tensor_cores":
        return dtype == "f32"
    if path == "tcgen05":
        return dtype == "f32" or D != 128
    return False


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("case", SWEEP, ids=[str(i) for i in range(len(SWEEP))])
def test_parity_sweep(svp, oracle_mod, case, path):
    """Every case through each kernel path (automatic choice, CUDA cores,
    warp-level tensor cores, tcgen05); a forced tensor path on data it cannot
    take must say so."""
    dtype, D, Hq, Hkv, q_len, lo, hi, n_sink, window, sp = case
    cfg = W.small_config(batch=5, num_q_heads=Hq, num_kv_heads=Hkv,
                         head_dim=D, q_len=q_len, dtype=dtype, ctx_min=lo,
                         ctx_max=hi, seed=100 + D + q_len + Hq)
    wl = W.make_attention(cfg, n_new=min(q_len, 2))
    if _unsupported(path, dtype, D):
        with pytest.raises(svp.SvpError) as e:
            _run_gpu(svp, wl, n_sink, window, split_pages=sp,
                     kernel_path=PATHS[path])
        assert e.value.status == -2
        return
    got = _run_gpu(svp, wl, n_sink, window, split_pages=sp,
                   kernel_path=PATHS[path])
    _compare(wl, got, _oracle(oracle_mod, wl, n_sink, window))


@pytest.mark.parametrize("path", [1, 2, 3])
@pytest.mark.parametrize("sp", [1, 2, 7, 64, 128])
def test_split_counts_agree(svp, oracle_mod, sp, path):
    """The same inputs under different split sizes (1 page per split up to
    128) all match the oracle: the log-sum-exp merge is exact."""
    cfg = W.small_config(batch=4, num_q_heads=8, num_kv_heads=2, head_dim=128,
                         q_len=2, ctx_min=2, ctx_max=900, seed=17)
    wl = W.make_attention(cfg)
    got = _run_gpu(svp, wl, 0, 0, split_pages=sp, kernel_path=path)
    _compare(wl, got, _oracle(oracle_mod, wl, 0, 0))


@pytest.mark.parametrize("path", [1, 2, 3])
@pytest.mark.parametrize("scale", [0.0, -0.07, 0.3])
def test_scale_sign(svp, oracle_mod, path, scale):
    """A zero, negative or large softmax scale (the kernels take the max of
    raw scores only for a positive scale)."""
    cfg = W.small_config(batch=3, num_q_heads=16, num_kv_heads=4,
                         head_dim=128, q_len=3, ctx_min=3, ctx_max=700,
                         seed=41)
    wl = W.make_attention(cfg, n_new=2)
    wl.scale = np.float32(scale)
    got = _run_gpu(svp, wl, 0, 0, kernel_path=path)
    _compare(wl, got, _oracle(oracle_mod, wl, 0, 0))


TWO_GROUPS = [
    # (Hq, Hkv, q_len, n_sink, window, split_pages): rows = Hq / Hkv * q_len
    (32, 8, 9, 0, 0, 0),     # 36 rows: the second group holds 4
    (32, 8, 9, 0, 0, 2),     # the same, split across CTAs
    (16, 1, 4, 0, 0, 1),     # exactly 64 rows, one page per split
    (8, 1, 9, 0, 0, 3),      # 72 rows: the second unit's second group is empty
    (32, 4, 6, 4, 37, 0),    # 48 rows under sinks + window
    (8, 2, 16, 0, 0, 7),     # 64 rows of one query position per 4 heads
]


@pytest.mark.parametrize("path", [0, 3])
@pytest.mark.parametrize("case", TWO_GROUPS,
                         ids=[str(i) for i in range(len(TWO_GROUPS))])
def test_tc_two_row_groups(svp, oracle_mod, case, path):
    """More than 32 rows per KV head: the tcgen05 kernel takes 64-row units
    whose two 32-row groups share every K/V tile; ragged and empty second
    groups, splits and a sink/window mask."""
    Hq, Hkv, q_len, n_sink, window, sp = case
    cfg = W.small_config(batch=4, num_q_heads=Hq, num_kv_heads=Hkv,
                         head_dim=128, q_len=q_len, ctx_min=q_len,
                         ctx_max=900, seed=400 + Hq + q_len + sp)
    wl = W.make_attention(cfg, n_new=min(q_len, 2))
    got = _run_gpu(svp, wl, n_sink, window, split_pages=sp, kernel_path=path)
    _compare(wl, got, _oracle(oracle_mod, wl, n_sink, window))


@pytest.mark.parametrize("path,q_len,Hq", [(1, 1, 4), (2, 1, 4), (2, 3, 8),
                                           (3, 1, 4), (3, 3, 8)])
def test_ring_layout_small(svp, oracle_mod, path, q_len, Hq):
    """A streaming cache in a ring of pages with NaN in every non-resident
    row: only sink and window rows may be read."""
    cfg = W.small_config(batch=3, num_q_heads=Hq, num_kv_heads=4,
                         head_dim=128, q_len=q_len, ctx_min=5000,
                         ctx_max=9000, n_sink=4, window=100, ring=True,
                         sink_key_scale=4.0, seed=23)
    wl = W.make_attention(cfg)
    got = _run_gpu(svp, wl, 4, 100, kernel_path=path)
    _compare(wl, got, _oracle(oracle_mod, wl, 4, 100))


def test_tiny_decode_config(svp, oracle_mod):
    """tiny-decode: fp32, every output compared, tolerance 1e-5."""
    wl = W.make_attention(W.CONFIGS["tiny-decode"])
    got = _run_gpu(svp, wl, 0, 0)
    _compare(wl, got, _oracle(oracle_mod, wl, 0, 0))


def _sampled_rows(wl, n, seed):
    rng = np.random.default_rng(seed)
    total = wl.cfg.batch * wl.q_len * wl.cfg.num_q_heads
    rows = rng.choice(total, size=min(n, total), replace=False)
    # always include the first and last row of every sequence
    per = wl.q_len * wl.cfg.num_q_heads
    edge = np.concatenate([np.arange(wl.cfg.batch) * per,
                           np.arange(1, wl.cfg.batch + 1) * per - 1])
    return np.unique(np.concatenate([rows, edge])).astype(np.int64)


@pytest.mark.parametrize("name,n_sink,window,n_rows", [
    ("decode-7b", 0, 0, 96),
    ("verify-gqa", 0, 0, 96),
    ("stream-sink-window", 4, 2044, 96),
    ("long-context-128k", 0, 0, 24),
    ("long-context-128k-verify", 0, 0, 24),
])
def test_full_size_configs_sampled(svp, oracle_mod, name, n_sink, window,
                                   n_rows):  # automatic path, as benchmarked
    """Each workload at full size, in the launch configuration the benchmark
    uses (automatic split size), compared on sampled rows."""
    wl = W.make_attention(W.CONFIGS[name], n_new=W.CONFIGS[name].q_len)
    got = _run_gpu(svp, wl, n_sink, window)
    rows = _sampled_rows(wl, n_rows, 1)
    ref = _oracle(oracle_mod, wl, n_sink, window, rows=rows)
    _compare(wl, got, ref, rows=rows)
    assert np.isfinite(got[0]).all() and np.isfinite(got[1]).all()


def test_empty_batch(svp):
    import torch
    dev = "cuda:0"
    q = torch.zeros((0, 1, 4, 64), dtype=torch.float32, device=dev)
    kc = torch.zeros((4, 4, 16, 64), dtype=torch.float32, device=dev)
    bt = torch.zeros((0, 1), dtype=torch.int32, device=dev)
    sl = torch.zeros((0,), dtype=torch.int32, device=dev)
    out, lse = svp.paged_decode_attention(q, kc, kc, bt, sl, q_len=1)
    assert out.shape == (0, 1, 4, 64) and svp.last_launch_count() == 0


@pytest.mark.parametrize("path", [1, 2, 3])
def test_bad_block_id_is_flagged_not_read(svp, path):
    """A block-table entry outside [0, num_blocks) is caught before any load:
    the device status reports it and nothing faults."""
    import torch
    cfg = W.small_config(batch=2, num_q_heads=4, num_kv_heads=4,
                         head_dim=128, ctx_min=40, ctx_max=40, seed=3)
    wl = W.make_attention(cfg)
    bt = wl.block_table.copy()
    bt[1, 1] = wl.num_blocks + 1000
    out, _ = svp.paged_decode_attention(
        to_dev(wl.q), to_dev(wl.k_cache), to_dev(wl.v_cache), to_dev(bt),
        to_dev(wl.seq_lens), q_len=1, kernel_path=path)
    torch.cuda.synchronize()
    assert svp.read_device_status() & 1
    assert svp.read_device_status() == 0  # read clears
    assert torch.isfinite(out.float()).all()


def test_bad_seq_len_is_flagged(svp):
    import torch
    cfg = W.small_config(batch=2, num_q_heads=4, num_kv_heads=4,
                         head_dim=128, ctx_min=40, ctx_max=40, seed=3)
    wl = W.make_attention(cfg)
    sl = wl.seq_lens.copy()
    sl[0] = 10 ** 6                    # beyond the table's reach
    svp.paged_decode_attention(to_dev(wl.q), to_dev(wl.k_cache),
                               to_dev(wl.v_cache), to_dev(wl.block_table),
                               to_dev(sl), q_len=1)
    torch.cuda.synchronize()
    assert svp.read_device_status() & 2


def test_repeated_calls_reuse_workspace(svp, oracle_mod):
    """Nothing in the workspace carries over between calls: ten calls in a
    row on the same workspace give identical results."""
    import torch
    cfg = W.small_config(batch=3, num_q_heads=8, num_kv_heads=2, head_dim=128,
                         q_len=2, ctx_min=100, ctx_max=800, seed=5)
    wl = W.make_attention(cfg)
    args = [to_dev(a) for a in (wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                                wl.seq_lens)]
    first = None
    for _ in range(10):
        out, lse = svp.paged_decode_attention(*args, q_len=2, split_pages=2)
        torch.cuda.synchronize()
        cur = (out.clone(), lse.clone())
        if first is None:
            first = cur
        assert torch.equal(first[0], cur[0]) and torch.equal(first[1], cur[1])
    _compare(wl, (out_as_f64(first[0]), first[1].cpu().numpy().astype(np.float64)),
             _oracle(oracle_mod, wl, 0, 0))


def test_workspace_shared_across_shapes(svp, oracle_mod):
    """One workspace, filled with junk first, serves calls of different
    shapes in any order: a small call, a call with many more split groups,
    then the small call again."""
    import torch
    ws = torch.full((64 << 20,), 0x5A, dtype=torch.uint8, device="cuda:0")
    shapes = [dict(batch=2, num_q_heads=8, num_kv_heads=2, q_len=2, ctx_max=900),
              dict(batch=24, num_q_heads=16, num_kv_heads=16, q_len=1, ctx_max=700),
              dict(batch=2, num_q_heads=8, num_kv_heads=2, q_len=2, ctx_max=900)]
    for i, kw in enumerate(shapes):
        cfg = W.small_config(head_dim=128, ctx_min=kw["q_len"], seed=40 + i,
                             **kw)
        wl = W.make_attention(cfg)
        out, lse = svp.paged_decode_attention(
            to_dev(wl.q), to_dev(wl.k_cache), to_dev(wl.v_cache),
            to_dev(wl.block_table), to_dev(wl.seq_lens), q_len=wl.q_len,
            scale=float(wl.scale), split_pages=3, workspace=ws)
        torch.cuda.synchronize()
        _compare(wl, (out_as_f64(out), lse.cpu().numpy().astype(np.float64)),
                 _oracle(oracle_mod, wl, 0, 0))


@pytest.mark.parametrize("path,batch", [(1, 4100), (3, 520)])
def test_many_sequences_span_launches(svp, oracle_mod, path, batch):
    """More sequences than one launch takes (4096 on CUDA cores, 512 on
    tcgen05): the call makes two attention launches on one workspace, each
    followed by its merge, with groups split over several CTAs in both;
    every output matches the oracle."""
    cfg = W.small_config(batch=batch, num_q_heads=4, num_kv_heads=1,
                         head_dim=128, q_len=2, ctx_min=2, ctx_max=70,
                         seed=61)
    wl = W.make_attention(cfg)
    got = _run_gpu(svp, wl, 0, 0, split_pages=1, kernel_path=path)
    assert svp.last_launch_count() == 4  # two attention + two merge launches
    _compare(wl, got, _oracle(oracle_mod, wl, 0, 0))


def test_many_sequences_span_launches_64_row_units(svp, oracle_mod):
    """The same beyond one tcgen05 launch with 40 query rows per kv head:
    64-row units, their split partials merged by two CTAs per group."""
    cfg = W.small_config(batch=520, num_q_heads=8, num_kv_heads=1,
                         head_dim=128, q_len=5, ctx_min=5, ctx_max=60,
                         seed=62)
    wl = W.make_attention(cfg, n_new=2)
    got = _run_gpu(svp, wl, 0, 0, split_pages=1, kernel_path=3)
    assert svp.last_launch_count() == 4  # two attention + two merge launches
    _compare(wl, got, _oracle(oracle_mod, wl, 0, 0))
