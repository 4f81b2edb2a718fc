"""paged_decode_attention_noalloc: the attention entry point for callers that
cannot allocate device memory (code running under CUDA-graph capture,
plug-ins whose host owns every allocation, loops where cudaMalloc would
synchronise the device).  Its split-K scratch is a fixed array inside the
library, so this test calls it through the C ABI with raw device pointers
and checks it against the allocating entry point and against the fp64
oracle, twice in a row (the array keeps the previous call's contents).
Kept in a file collected last."""
import ctypes

import numpy as np
import pytest

from helpers import out_as_f64, to_dev
from spec_verify_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-5}
LSE_TOL = 1e-3


@pytest.fixture(scope="module")
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from spec_verify_paged_gb300 import binding
    return binding.load_library()


CASES = [
    # decode, MHA, several splits per sequence (CUDA-core path)
    dict(batch=6, num_q_heads=8, num_kv_heads=8, head_dim=128, q_len=1,
         dtype="bf16", ctx_min=1, ctx_max=1500, split_pages=4, path=0),
    # verify, GQA 4, q_len 5, tensor-core path, sinks + window
    dict(batch=5, num_q_heads=16, num_kv_heads=4, head_dim=128, q_len=5,
         dtype="bf16", ctx_min=5, ctx_max=2000, split_pages=0, path=0,
         n_sink=4, window=300),
    # fp32, head_dim 64
    dict(batch=3, num_q_heads=4, num_kv_heads=2, head_dim=64, q_len=2,
         dtype="f32", ctx_min=2, ctx_max=600, split_pages=2, path=1),
]


@pytest.mark.parametrize("case", CASES, ids=["decode", "verify", "fp32"])
def test_noalloc_matches_allocating_call_twice(lib, oracle_mod, case):
    import torch
    import spec_verify_paged_gb300 as svp
    from spec_verify_paged_gb300 import binding
    case = dict(case)
    sp, path = case.pop("split_pages"), case.pop("path")
    n_sink, window = case.pop("n_sink", 0), case.pop("window", 0)
    cfg = W.small_config(seed=77, **case)
    wl = W.make_attention(cfg)
    q, kc, vc = to_dev(wl.q), to_dev(wl.k_cache), to_dev(wl.v_cache)
    bt, sl = to_dev(wl.block_table), to_dev(wl.seq_lens)
    ref_out, ref_lse = svp.paged_decode_attention(
        q, kc, vc, bt, sl, q_len=wl.q_len, n_sink=n_sink, window=window,
        scale=float(wl.scale), split_pages=sp, kernel_path=path)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle_mod.paged_attention(
        wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.seq_lens, wl.q_len,
        n_sink, window, wl.scale)
    dims = binding.make_dims(q.shape, kc, bt, binding._dtype_code(q), None,
                             sp, path)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        st = lib.paged_decode_attention_noalloc(
            ctypes.byref(dims), q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
            bt.data_ptr(), sl.data_ptr(), wl.q_len, n_sink, window,
            float(wl.scale), out.data_ptr(), lse.data_ptr(), stream)
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
        err = (out.float() - ref_out.float()).abs().max().item()
        lerr = (lse - ref_lse).abs().max().item()
        assert err <= TOL[cfg.dtype], (call, err)
        assert lerr <= LSE_TOL, (call, lerr)
        # and against the oracle itself
        oerr = np.abs(out_as_f64(out) - o_ref).max()
        olerr = np.abs(lse.cpu().numpy().astype(np.float64) - l_ref).max()
        assert oerr <= TOL[cfg.dtype], (call, oerr)
        assert olerr <= LSE_TOL, (call, olerr)
    assert svp.read_device_status() == 0


def test_scratch_holds_the_largest_plans(lib):
    """Every plan on this GPU fits the fixed array: the split scratch is two
    partial slots per CTA of the persistent grid, whatever the batch, so
    SVP_ERR_WORKSPACE cannot occur here (the check guards GPUs with more
    SMs).  Sizes only: nothing is launched."""
    from spec_verify_paged_gb300 import binding
    cap = lib.paged_decode_workspace_size  # bytes each plan needs
    for path, rows_q_len, hq, hkv, dtype in [
            (1, 1, 64, 64, 0), (1, 16, 64, 8, 1), (2, 16, 64, 4, 1),
            (3, 16, 64, 8, 1), (0, 4, 64, 8, 1)]:
        d = binding.SvpDims()
        d.batch, d.num_q_heads, d.num_kv_heads, d.head_dim = 4096, hq, hkv, 128
        d.block_size, d.max_blocks_per_seq, d.num_blocks = 16, 8192, 1 << 20
        d.dtype, d.split_pages, d.kernel_path = dtype, 1, path
        need = cap(ctypes.byref(d), rows_q_len, 0, 0)
        assert 0 < need <= 32 << 20, (path, need)
