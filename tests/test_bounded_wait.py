"""The bounded-wait path of the attention kernels, run on the GPU without a
fault or a hang.

A test build of the library (libsvp_stalltest.so, a separate copy with its
own kernels and device status word) shortens the pipeline waits to 20 ms and
makes each CTA's producer stop after a few copies and wait on a barrier that
nothing arrives on.  Every role's wait then runs out: the kernel raises
SVP_DEV_TIMEOUT, drains the copies and MMAs it started (those waits keep the
2 s limit), frees its tensor memory and returns.  The test checks that the
call returns promptly with the flag raised, and that the next call of the
normal library in the same process, on the same inputs, matches the fp64
oracle: the context is intact."""
import ctypes
import time

import numpy as np
import pytest

from helpers import out_as_f64, to_dev
from spec_verify_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SVP_DEV_TIMEOUT = 8
STALL_DEFINES = ["SVP_WAIT_NS=20000000ull", "SVP_TEST_STALL_AFTER=2"]
# 64 pages per CTA: every CTA's slice is longer than the producer's two
# copies (pages, or 8-page tiles) before it stalls
SPLIT_PAGES = 64


@pytest.fixture(scope="module")
def libs():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from spec_verify_paged_gb300 import binding, build
    stall = binding.load_library(build.build_variant("stalltest", STALL_DEFINES))
    return binding.load_library(), stall


CASES = [
    # CUDA-core kernel: MHA decode, one row per kv head
    dict(batch=4, num_q_heads=8, num_kv_heads=8, head_dim=128, q_len=1,
         dtype="bf16", ctx_min=300, ctx_max=900, path=1),
    # tcgen05 kernel: 20 rows per kv head (one 32-row unit)
    dict(batch=4, num_q_heads=16, num_kv_heads=4, head_dim=128, q_len=5,
         dtype="bf16", ctx_min=600, ctx_max=1500, path=3),
    # tcgen05 kernel, 64-row units (two 32-row groups sharing each tile)
    dict(batch=3, num_q_heads=32, num_kv_heads=2, head_dim=128, q_len=3,
         dtype="bf16", ctx_min=600, ctx_max=1500, path=3),
]


def _call(lib, wl, path, q, kc, vc, bt, sl, out, lse, ws):
    import torch
    from spec_verify_paged_gb300 import binding
    dims = binding.make_dims(q.shape, kc, bt, binding._dtype_code(q), ws,
                             SPLIT_PAGES, path)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.paged_decode_attention(
        ctypes.byref(dims), q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
        bt.data_ptr(), sl.data_ptr(), wl.q_len, 0, 0, float(wl.scale),
        out.data_ptr(), lse.data_ptr(), stream)


def _flags(lib):
    import torch
    f = ctypes.c_int(0)
    st = lib.svp_read_device_status(
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
        ctypes.byref(f))
    assert st == 0
    return f.value


@pytest.mark.parametrize("case", CASES, ids=["cuda-cores", "tcgen05", "tcgen05-64"])
def test_timeout_raises_flag_and_context_survives(libs, oracle_mod, case):
    import torch
    normal, stall = libs
    case = dict(case)
    path = case.pop("path")
    cfg = W.small_config(seed=88, **case)
    wl = W.make_attention(cfg)
    q, kc, vc = to_dev(wl.q), to_dev(wl.k_cache), to_dev(wl.v_cache)
    bt, sl = to_dev(wl.block_table), to_dev(wl.seq_lens)
    lse = torch.empty(wl.q.shape[:3], dtype=torch.float32, device="cuda:0")
    out = torch.empty_like(q)
    from spec_verify_paged_gb300 import binding
    dims = binding.make_dims(q.shape, kc, bt, binding._dtype_code(q), None,
                             SPLIT_PAGES, path)
    need = stall.paged_decode_workspace_size(ctypes.byref(dims), wl.q_len, 0, 0)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda:0")
    assert _flags(stall) == 0
    # the stalled call: every wait runs out after 20 ms, the kernel drains
    # and returns
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert _call(stall, wl, path, q, kc, vc, bt, sl, out, lse, ws) == 0
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    flags = _flags(stall)
    assert flags & SVP_DEV_TIMEOUT, flags
    assert dt < 1.5, f"the stalled call took {dt:.2f} s"
    # the normal library on the same inputs, same process: correct results
    out.fill_(float("nan"))
    lse.fill_(float("nan"))
    assert _call(normal, wl, path, q, kc, vc, bt, sl, out, lse, ws) == 0
    torch.cuda.synchronize()
    assert _flags(normal) == 0
    o_ref, l_ref = oracle_mod.paged_attention(
        wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.seq_lens, wl.q_len,
        0, 0, wl.scale)
    assert np.abs(out_as_f64(out) - o_ref).max() <= 2e-2
    assert np.abs(lse.cpu().numpy().astype(np.float64) - l_ref).max() <= 1e-3
