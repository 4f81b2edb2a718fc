"""The C ABI without a GPU: the library builds, loads, exports every symbol
include/svp.h declares, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from spec_verify_paged_gb300 import binding, build
    build.build()
    return binding.load_library()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "svp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\([^;{]*\)\s*;", src)
    return sorted(set(n for n in names if n not in ("sizeof",)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert {"paged_decode_attention", "spec_accept", "kv_append"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} missing from libsvp.so"


def test_binding_covers_the_header():
    from spec_verify_paged_gb300 import binding
    assert set(_declared_functions()) == set(binding.EXPORTED)


def _dims(**kw):
    from spec_verify_paged_gb300.binding import SvpDims
    d = SvpDims()
    base = dict(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128,
                block_size=16, max_blocks_per_seq=4, num_blocks=8, dtype=1,
                split_pages=0)
    base.update(kw)
    for k, v in base.items():
        setattr(d, k, v)
    return d


P = ctypes.c_void_p(0x1000)  # never dereferenced: every call below fails its checks


@pytest.mark.parametrize("kw,q_len,n_sink,window,scale,expect", [
    (dict(head_dim=96), 1, 0, 0, 0.1, -2),
    (dict(block_size=32), 1, 0, 0, 0.1, -2),
    (dict(num_q_heads=6, num_kv_heads=4), 1, 0, 0, 0.1, -1),
    (dict(dtype=7), 1, 0, 0, 0.1, -1),
    (dict(batch=-1), 1, 0, 0, 0.1, -1),
    (dict(batch=70000), 1, 0, 0, 0.1, -2),
    ({}, 0, 0, 0, 0.1, -1),
    ({}, 17, 0, 0, 0.1, -2),
    ({}, 1, -1, 0, 0.1, -1),
    ({}, 1, 0, -3, 0.1, -1),
    ({}, 1, 0, 0, float("nan"), -1),
    ({}, 1, 0, 0, float("inf"), -1),
])
def test_attention_rejects_bad_arguments(lib, kw, q_len, n_sink, window, scale,
                                         expect):
    d = _dims(**kw)
    st = lib.paged_decode_attention(ctypes.byref(d), P, P, P, P, P, q_len,
                                    n_sink, window, scale, P, P, None)
    assert st == expect
    assert lib.svp_last_launch_count() == 0


def test_attention_null_pointers(lib):
    d = _dims()
    assert lib.paged_decode_attention(None, P, P, P, P, P, 1, 0, 0, 0.1, P, P,
                                      None) == -1
    assert lib.paged_decode_attention(ctypes.byref(d), None, P, P, P, P, 1, 0,
                                      0, 0.1, P, P, None) == -1
    assert lib.paged_decode_attention(ctypes.byref(d), P, P, P, P, P, 1, 0, 0,
                                      0.1, P, None, None) == -1


def test_tree_attention_needs_a_mask(lib):
    d = _dims()
    assert lib.paged_tree_attention(ctypes.byref(d), P, P, P, P, P, 3, None,
                                    0.1, P, P, None) == -1
    # misaligned mask pointer
    assert lib.paged_tree_attention(ctypes.byref(d), P, P, P, P, P, 3, 0x1002,
                                    0.1, P, P, None) == -1
    # q_len beyond the tree limit
    assert lib.paged_tree_attention(ctypes.byref(d), P, P, P, P, P, 17, P, 0.1,
                                    P, P, None) == -2


def test_fp8_cache_needs_positive_scales(lib):
    d = _dims(dtype=2)                       # k_scale = v_scale = 0
    assert lib.paged_decode_attention(ctypes.byref(d), P, P, P, P, P, 1, 0, 0,
                                      0.1, P, P, None) == -1
    assert lib.kv_append(ctypes.byref(d), P, P, P, P, P, P, 1, None) == -1
    d = _dims(dtype=2, k_scale=float("inf"), v_scale=1.0)
    assert lib.paged_decode_workspace_size(ctypes.byref(d), 1, 0, 0) == 0
    d = _dims(dtype=2, k_scale=0.03, v_scale=0.03)
    assert lib.paged_decode_workspace_size(ctypes.byref(d), 1, 0, 0) > 0


def test_attention_empty_batch_is_a_no_op(lib):
    d = _dims(batch=0)
    assert lib.paged_decode_attention(ctypes.byref(d), None, None, None, None,
                                      None, 1, 0, 0, 0.1, None, None, None) == 0
    assert lib.svp_last_launch_count() == 0


def test_workspace_too_small(lib):
    d = _dims()
    d.workspace = P
    d.workspace_bytes = 16
    # the plan is made before any launch; a short workspace is refused
    st = lib.paged_decode_attention(ctypes.byref(d), P, P, P, P, P, 1, 0, 0,
                                    0.1, P, P, None)
    assert st in (-4, -3)  # -3 only where no device can be queried


def test_workspace_size_grows_with_work(lib):
    """Header + one split descriptor and two partial slots per CTA of the
    grid: more work never needs less, a window never needs more."""
    small = lib.paged_decode_workspace_size(ctypes.byref(_dims()), 1, 0, 0)
    many = dict(batch=4096, max_blocks_per_seq=512)  # same heads and rows
    big = lib.paged_decode_workspace_size(ctypes.byref(_dims(**many)), 1, 0, 0)
    win = lib.paged_decode_workspace_size(ctypes.byref(_dims(**many)), 1, 4, 64)
    assert 0 < small <= big and win <= big
    # header (256) + descriptors (256-aligned) + one slot pair of head_dim
    assert small >= 256 + 256 + 2 * 128 * 4
    assert lib.paged_decode_workspace_size(None, 1, 0, 0) == 0
    assert lib.paged_decode_workspace_size(ctypes.byref(_dims(head_dim=80)),
                                           1, 0, 0) == 0


@pytest.mark.parametrize("args,expect", [
    ((2, 0, 100), -1), ((2, 4, 1), -1), ((-1, 4, 100), -1),
    ((2, 16, 100), -2), ((70000, 4, 100), -2), ((2, 4, 8 * 40000 + 1), -2),
])
def test_accept_rejects_bad_sizes(lib, args, expect):
    assert lib.spec_accept(*args, P, P, P, P, P, P, None) == expect


@pytest.mark.parametrize("args,expect", [
    ((-1, 4, 100), -1), ((2, 0, 100), -1), ((2, 4, 1), -1),
    ((2, 17, 100), -2), ((70000, 4, 100), -2), ((2, 4, 400000), -2),
])
def test_accept_tree_rejects_bad_sizes(lib, args, expect):
    assert lib.spec_accept_tree(*args, *([P] * 8), None) == expect


def test_accept_tree_null_pointer_and_empty_batch(lib):
    ptrs = [P] * 8
    ptrs[3] = None  # uniforms
    assert lib.spec_accept_tree(2, 4, 100, *ptrs, None) == -1
    assert lib.spec_accept_tree(0, 4, 100, *([None] * 8), None) == 0
    assert lib.svp_last_launch_count() == 0


def test_accept_ex_checks_its_options(lib):
    from spec_verify_paged_gb300.binding import SvpAcceptOpts
    bad_t = SvpAcceptOpts(0.0, None, 0)
    assert lib.spec_accept_ex(2, 4, 100, P, P, P, P, ctypes.byref(bad_t), P, P,
                              None) == -1
    nan_t = SvpAcceptOpts(float("nan"), None, 0)
    assert lib.spec_accept_ex(2, 4, 100, P, P, P, P, ctypes.byref(nan_t), P, P,
                              None) == -1
    odd_mask = SvpAcceptOpts(1.0, 0x1002, 0)
    assert lib.spec_accept_ex(2, 4, 100, P, P, P, P, ctypes.byref(odd_mask), P,
                              P, None) == -1
    # greedy ignores the temperature; an empty batch launches nothing
    greedy = SvpAcceptOpts(0.0, None, 1)
    assert lib.spec_accept_ex(0, 4, 100, P, P, P, P, ctypes.byref(greedy), P,
                              P, None) == 0
    assert lib.spec_accept_ex(2, 16, 100, P, P, P, P, None, P, P, None) == -2


def test_step_runner_rejects_bad_descriptions(lib):
    from spec_verify_paged_gb300.binding import SvpStepDesc
    h = ctypes.c_void_p()
    assert lib.svp_step_create(None, ctypes.byref(h)) == -1
    d = SvpStepDesc(_dims(batch=0), 5, 0, 0, 0.1, P, P, 4, 100)
    assert lib.svp_step_create(ctypes.byref(d), ctypes.byref(h)) == -1
    d = SvpStepDesc(_dims(), 5, 0, 0, 0.1, P, P, 3, 100)   # K != q_len - 1
    assert lib.svp_step_create(ctypes.byref(d), ctypes.byref(h)) == -1
    assert lib.svp_step_launch(None, 0) == -1
    assert lib.svp_step_host_buffer(None, 0, 0, None) is None


@pytest.mark.parametrize("q_len,n_sink,window,num_draft,temp,greedy,mask,tree,expect", [
    (1, 0, 0, 0, 1.0, 1, 0, 0, -1),     # greedy without drafts
    (1, 0, 0, 0, 0.7, 0, 0, 0, -1),     # a temperature without drafts
    (5, 0, 0, 4, -0.5, 0, 0, 0, -1),    # negative temperature
    (7, 0, 0, 6, 1.0, 0, 0, 7, -1),     # a tree with chain drafts
    (7, 0, 0, 0, 1.0, 0, 0, 5, -1),     # tree_nodes != q_len
    (7, 0, 16, 0, 1.0, 0, 0, 7, -1),    # a tree under a window
    (7, 4, 0, 0, 1.0, 0, 0, 7, -1),     # a tree with sinks
    (7, 0, 0, 0, 1.0, 1, 0, 7, -1),     # a tree with epilogue options
    (7, 0, 0, 0, 1.0, 0, 1, 7, -1),
    (17, 0, 0, 0, 1.0, 0, 0, 17, -2),   # more nodes than the kernels take
])
def test_step_runner_checks_epilogue_and_tree_options(lib, q_len, n_sink, window,
                                                      num_draft, temp, greedy,
                                                      mask, tree, expect):
    """Epilogue options need draft chains; a draft tree needs tree_nodes =
    q_len, no chain drafts, sinks, window or options; all checked before
    anything touches the GPU."""
    from spec_verify_paged_gb300.binding import SvpStepDesc
    h = ctypes.c_void_p()
    d = SvpStepDesc(_dims(), q_len, n_sink, window, 0.1, P, P, num_draft, 100,
                    temp, greedy, mask, tree)
    assert lib.svp_step_create(ctypes.byref(d), ctypes.byref(h)) == expect


def test_accept_null_pointer(lib):
    assert lib.spec_accept(2, 4, 100, P, None, P, P, P, P, None) == -1
    assert lib.spec_accept(0, 4, 100, None, None, None, None, None, None,
                           None) == 0


def test_append_rejects_bad_arguments(lib):
    d = _dims()
    assert lib.kv_append(ctypes.byref(d), P, P, P, P, P, P, -1, None) == -1
    assert lib.kv_append(ctypes.byref(d), P, P, P, P, P, P, 65, None) == -2
    assert lib.kv_append(ctypes.byref(_dims(head_dim=32)), P, P, P, P, P, P, 1,
                         None) == -2
    assert lib.kv_append(ctypes.byref(d), None, P, P, P, P, P, 1, None) == -1
    assert lib.kv_append(ctypes.byref(d), P, P, P, P, P, P, 0, None) == 0


@pytest.mark.parametrize("which", range(4))
def test_append_rejects_unaligned_rows(lib, which):
    """The append moves rows as 16-byte vectors: a pointer that is not
    16-byte aligned (an offset view) is refused on the host, before any
    launch, instead of faulting on the device."""
    d = _dims()
    ptrs = [P, P, P, P]
    ptrs[which] = ctypes.c_void_p(P.value + 2)
    assert lib.kv_append(ctypes.byref(d), *ptrs, P, P, 1, None) == -1
    assert lib.svp_last_launch_count() == 0


def test_noalloc_fallback_splits_need_no_more_scratch(lib):
    """The no-alloc entry point retries a plan that does not fit its fixed
    array with 64 and then 128 pages per CTA; those plans never need more
    scratch than the automatic one (fewer or equal partial slots)."""
    for kw in (dict(), dict(batch=4096, max_blocks_per_seq=8192),
               dict(batch=64, num_q_heads=64, num_kv_heads=8,
                    max_blocks_per_seq=8192)):
        base = lib.paged_decode_workspace_size(ctypes.byref(_dims(**kw)), 1, 0, 0)
        assert base > 0
        for pps in (64, 128):
            d = _dims(**kw)
            d.split_pages = pps
            n = lib.paged_decode_workspace_size(ctypes.byref(d), 1, 0, 0)
            assert 0 < n <= base, (kw, pps, n, base)


def test_status_strings(lib):
    assert lib.svp_status_string(0) == b"SVP_OK"
    assert lib.svp_status_string(-4) == b"SVP_ERR_WORKSPACE"
    assert lib.svp_status_string(5) == b"SVP_UNKNOWN_STATUS"


def test_product_path_fails_loudly_without_the_library(tmp_path):
    """No CPU fallback: a missing library is an error, not a slow path."""
    from spec_verify_paged_gb300 import binding
    with pytest.raises(RuntimeError):
        binding.load_library.__wrapped__(str(tmp_path / "nope.so")) \
            if hasattr(binding.load_library, "__wrapped__") else \
            _load_missing(binding, tmp_path)


def _load_missing(binding, tmp_path):
    saved = binding._lib
    binding._lib = None
    try:
        binding.load_library(str(tmp_path / "missing.so"))
    finally:
        binding._lib = saved
