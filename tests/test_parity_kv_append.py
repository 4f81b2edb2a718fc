"""GPU kv_append vs the oracle: a byte copy, so bit-exact."""
import numpy as np
import pytest

from helpers import to_dev, to_host
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


@pytest.mark.parametrize("dtype,D,n_new", [("bf16", 128, 1), ("bf16", 128, 5),
                                           ("f32", 64, 3), ("bf16", 64, 16),
                                           ("f32", 128, 1)])
def test_append_bit_exact(svp, oracle_mod, dtype, D, n_new):
    import torch
    cfg = W.small_config(batch=7, num_q_heads=8, num_kv_heads=4, head_dim=D,
                         q_len=1, dtype=dtype, ctx_min=n_new, ctx_max=300,
                         seed=D + n_new)
    wl = W.make_attention(cfg, n_new=n_new, spare_blocks=3)
    kc, vc = to_dev(wl.k_cache), to_dev(wl.v_cache)
    svp.kv_append(to_dev(wl.k_new), to_dev(wl.v_new), kc, vc,
                  to_dev(wl.block_table), to_dev(wl.seq_lens))
    torch.cuda.synchronize()
    k_ref, v_ref = oracle_mod.kv_append(wl.k_new, wl.v_new, wl.k_cache,
                                        wl.v_cache, wl.block_table,
                                        wl.seq_lens)
    view = np.uint16 if dtype == "bf16" else np.uint32
    assert np.array_equal(to_host(kc).view(view), k_ref.view(view))
    assert np.array_equal(to_host(vc).view(view), v_ref.view(view))
    assert svp.read_device_status() == 0


def test_append_bad_block_flagged(svp):
    import torch
    cfg = W.small_config(batch=2, num_q_heads=4, num_kv_heads=4, head_dim=128,
                         ctx_min=20, ctx_max=20, seed=1)
    wl = W.make_attention(cfg, n_new=1)
    bt = wl.block_table.copy()
    bt[0, 1] = -7
    kc = to_dev(wl.k_cache)
    before = to_host(kc).copy()
    svp.kv_append(to_dev(wl.k_new), to_dev(wl.v_new), kc, to_dev(wl.v_cache),
                  to_dev(bt), to_dev(wl.seq_lens))
    torch.cuda.synchronize()
    assert svp.read_device_status() & 1
    after = to_host(kc)
    # sequence 1 was written, sequence 0 was skipped
    assert (after.view(np.uint16) != before.view(np.uint16)).sum() == 4 * 128
