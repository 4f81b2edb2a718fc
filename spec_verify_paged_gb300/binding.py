"""Thin ctypes binding of libsvp.so (include/svp.h).

Argument marshalling only: shape/dtype/device checks, raw device pointers,
the current CUDA stream, and a zero-filled workspace tensor kept per device.
Every step of the computation runs in the library's CUDA kernels; there is
no fallback of any kind -- if libsvp.so is missing or no GPU is present the
calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import numpy as np

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsvp.so")

SVP_OK, SVP_ERR_INVALID_ARG, SVP_ERR_UNSUPPORTED, SVP_ERR_CUDA, SVP_ERR_WORKSPACE = (
    0, -1, -2, -3, -4)
SVP_F32, SVP_BF16, SVP_FP8_E4M3 = 0, 1, 2
PATH_AUTO, PATH_CUDA_CORES, PATH_TENSOR_CORES, PATH_TCGEN05 = 0, 1, 2, 3
DEV_BAD_BLOCK_ID, DEV_BAD_SEQ_LEN, DEV_BAD_TOKEN, DEV_TIMEOUT = 1, 2, 4, 8
EXPORTED = ("paged_decode_attention", "paged_decode_attention_noalloc",
            "paged_tree_attention",
            "paged_decode_workspace_size",
            "kv_append", "spec_accept", "spec_accept_ex", "spec_accept_tree",
            "svp_read_device_status",
            "svp_step_create", "svp_step_host_buffer", "svp_step_launch",
            "svp_step_wait", "svp_step_stream", "svp_step_destroy",
            "svp_status_string", "svp_last_launch_count")


class SvpDims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("num_q_heads", ctypes.c_int),
                ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("block_size", ctypes.c_int),
                ("max_blocks_per_seq", ctypes.c_int),
                ("num_blocks", ctypes.c_int), ("dtype", ctypes.c_int),
                ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t),
                ("split_pages", ctypes.c_int),
                ("kernel_path", ctypes.c_int),
                ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float)]


class SvpAcceptOpts(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("allowed", ctypes.c_void_p),
                ("greedy", ctypes.c_int)]


class SvpStepDesc(ctypes.Structure):
    _fields_ = [("dims", SvpDims), ("q_len", ctypes.c_int),
                ("n_sink", ctypes.c_int), ("window", ctypes.c_int),
                ("scale", ctypes.c_float), ("k_cache", ctypes.c_void_p),
                ("v_cache", ctypes.c_void_p), ("num_draft", ctypes.c_int),
                ("vocab", ctypes.c_int), ("temperature", ctypes.c_float),
                ("greedy", ctypes.c_int), ("use_mask", ctypes.c_int),
                ("tree_nodes", ctypes.c_int)]


STEP_FIELDS = ("q", "k_new", "v_new", "block_table", "seq_lens",
               "target_logits", "draft_logits", "draft_tokens", "uniforms",
               "out", "lse", "out_tokens", "n_accepted", "allowed",
               "tree_mask", "parents", "node_tokens", "out_nodes")


class SvpError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn} returned {status} ({msg})")
        self.status = status


_lock = threading.Lock()
_lib = None


_variants = {}


def load_library(path: str = LIB_PATH):
    """Load libsvp.so (raises if it has not been built).  Another path loads
    a separately built copy of the library (its own kernels and device
    state), e.g. a test build."""
    global _lib
    with _lock:
        if path == LIB_PATH and _lib is not None:
            return _lib
        if path in _variants:
            return _variants[path]
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        dims_p = ctypes.POINTER(SvpDims)
        lib.paged_decode_attention.argtypes = [dims_p, vp, vp, vp, vp, vp, i32,
                                               i32, i32, f32, vp, vp, vp]
        lib.paged_decode_attention.restype = i32
        lib.paged_decode_attention_noalloc.argtypes = [dims_p, vp, vp, vp, vp,
                                                       vp, i32, i32, i32, f32,
                                                       vp, vp, vp]
        lib.paged_decode_attention_noalloc.restype = i32
        lib.paged_tree_attention.argtypes = [dims_p, vp, vp, vp, vp, vp, i32,
                                             vp, f32, vp, vp, vp]
        lib.paged_tree_attention.restype = i32
        lib.paged_decode_workspace_size.argtypes = [dims_p, i32, i32, i32]
        lib.paged_decode_workspace_size.restype = sz
        lib.kv_append.argtypes = [dims_p, vp, vp, vp, vp, vp, vp, i32, vp]
        lib.kv_append.restype = i32
        lib.spec_accept.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
        lib.spec_accept.restype = i32
        lib.spec_accept_ex.argtypes = ([i32, i32, i32] + [vp] * 4 +
                                       [ctypes.POINTER(SvpAcceptOpts)] +
                                       [vp] * 3)
        lib.spec_accept_ex.restype = i32
        lib.spec_accept_tree.argtypes = [i32, i32, i32] + [vp] * 9
        lib.spec_accept_tree.restype = i32
        lib.svp_step_create.argtypes = [ctypes.POINTER(SvpStepDesc),
                                         ctypes.POINTER(vp)]
        lib.svp_step_create.restype = i32
        lib.svp_step_host_buffer.argtypes = [vp, i32, i32, ctypes.POINTER(sz)]
        lib.svp_step_host_buffer.restype = vp
        lib.svp_step_launch.argtypes = [vp, i32]
        lib.svp_step_launch.restype = i32
        lib.svp_step_wait.argtypes = [vp, i32]
        lib.svp_step_wait.restype = i32
        lib.svp_step_stream.argtypes = [vp]
        lib.svp_step_stream.restype = vp
        lib.svp_step_destroy.argtypes = [vp]
        lib.svp_step_destroy.restype = i32
        lib.svp_read_device_status.argtypes = [vp, ctypes.POINTER(i32)]
        lib.svp_read_device_status.restype = i32
        lib.svp_status_string.argtypes = [i32]
        lib.svp_status_string.restype = ctypes.c_char_p
        lib.svp_last_launch_count.argtypes = []
        lib.svp_last_launch_count.restype = i32
        if path == LIB_PATH:
            _lib = lib
        else:
            _variants[path] = lib
        return lib


def _check(fn, status):
    if status != SVP_OK:
        msg = _lib.svp_status_string(status).decode()
        raise SvpError(fn, status, msg)


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SVP_F32
    if t.dtype == torch.bfloat16:
        return SVP_BF16
    raise TypeError(f"q/k/v must be float32 or bfloat16, got {t.dtype}")


_FP8_TYPES = (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8))


def _cache_code(k_cache, q_dtype):
    """dtype code of a call: the cache's; an FP8 E4M3 cache (uint8 codes or
    float8_e4m3fn) pairs with bf16 q / out / new rows."""
    if k_cache.dtype in _FP8_TYPES:
        _need(q_dtype == torch.bfloat16,
              "an FP8 cache takes bf16 q, out and new rows")
        return SVP_FP8_E4M3
    _need(k_cache.dtype == q_dtype, "q and the caches must share a dtype")
    return _dtype_code(k_cache)


def _need(cond, what):
    if not cond:
        raise ValueError(what)


def _cuda_contig(t, name):
    _need(t.is_cuda, f"{name} must be a CUDA tensor")
    _need(t.is_contiguous(), f"{name} must be contiguous")


def make_dims(q_shape, k_cache, block_table, dtype_code, workspace=None,
              split_pages=0, kernel_path=0, k_scale=1.0, v_scale=1.0):
    B, _, Hq, D = q_shape
    nb, Hkv, bs, D2 = k_cache.shape
    d = SvpDims()
    d.batch, d.num_q_heads, d.num_kv_heads, d.head_dim = B, Hq, Hkv, D
    d.block_size, d.max_blocks_per_seq, d.num_blocks = bs, block_table.shape[1], nb
    d.dtype = dtype_code
    d.split_pages = int(split_pages)
    d.kernel_path = int(kernel_path)
    d.k_scale = float(k_scale)
    d.v_scale = float(v_scale)
    if workspace is not None:
        d.workspace = ctypes.c_void_p(workspace.data_ptr())
        d.workspace_bytes = workspace.numel() * workspace.element_size()
    return d


_ws_cache: dict = {}


def workspace_for(dims: SvpDims, q_len: int, n_sink: int, window: int,
                  device) -> torch.Tensor:
    """A workspace of at least the required size, kept per device and
    reused (calls that share it must not overlap on the GPU).  None for a
    request the library rejects."""
    lib = load_library()
    need = int(lib.paged_decode_workspace_size(ctypes.byref(dims), q_len,
                                               n_sink, window))
    if need == 0:  # an invalid request: the call itself reports the status
        return None
    key = torch.device(device).index or 0
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(need, dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def paged_decode_attention(q, k_cache, v_cache, block_table, seq_lens,
                           q_len=None, n_sink=0, window=0, scale=None,
                           out=None, lse=None, workspace=None, split_pages=0,
                           kernel_path=PATH_AUTO, stream=None, k_scale=1.0,
                           v_scale=1.0):
    """out [B, q_len, Hq, D] (q's dtype) and lse [B, q_len, Hq] fp32 of paged
    decode/verify attention (include/svp.h: paged_decode_attention).  FP8
    E4M3 caches (uint8 codes or float8_e4m3fn) take bf16 q and their
    k_scale / v_scale."""
    return _attention(q, k_cache, v_cache, block_table, seq_lens, q_len,
                      n_sink, window, None, scale, out, lse, workspace,
                      split_pages, kernel_path, stream, k_scale, v_scale)


def paged_tree_attention(q, k_cache, v_cache, block_table, seq_lens,
                         tree_mask, scale=None, out=None, lse=None,
                         workspace=None, split_pages=0, kernel_path=PATH_AUTO,
                         stream=None, k_scale=1.0, v_scale=1.0):
    """Draft-tree verify attention (include/svp.h: paged_tree_attention).
    tree_mask: int32 (or uint32) [B, q_len] on the GPU, bit k of entry
    (b, i) set iff node k is an ancestor of node i or i itself."""
    _cuda_contig(tree_mask, "tree_mask")
    _need(tree_mask.dtype in (torch.int32, getattr(torch, "uint32", torch.int32))
          and tuple(tree_mask.shape) == tuple(q.shape[:2]),
          "tree_mask must be int32/uint32 [B, q_len]")
    return _attention(q, k_cache, v_cache, block_table, seq_lens, None, 0, 0,
                      tree_mask, scale, out, lse, workspace, split_pages,
                      kernel_path, stream, k_scale, v_scale)


def _attention(q, k_cache, v_cache, block_table, seq_lens, q_len, n_sink,
               window, tree_mask, scale, out, lse, workspace, split_pages,
               kernel_path, stream, k_scale=1.0, v_scale=1.0):
    lib = load_library()
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (block_table, "block_table"), (seq_lens, "seq_lens")):
        _cuda_contig(t, n)
    code = _cache_code(k_cache, q.dtype)
    _need(v_cache.dtype == k_cache.dtype, "k_cache and v_cache must share a dtype")
    _need(k_cache.shape == v_cache.shape and k_cache.dim() == 4,
          "k_cache/v_cache must be [num_blocks, Hkv, block_size, D]")
    _need(block_table.dtype == torch.int32 and block_table.dim() == 2,
          "block_table must be int32 [B, max_blocks]")
    _need(seq_lens.dtype == torch.int32 and seq_lens.dim() == 1,
          "seq_lens must be int32 [B]")
    B, ql, Hq, D = q.shape
    q_len = ql if q_len is None else q_len
    _need(ql == q_len, "q.shape[1] must equal q_len")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, q_len, Hq), dtype=torch.float32, device=q.device)
    _cuda_contig(out, "out")
    _cuda_contig(lse, "lse")
    dims = make_dims(q.shape, k_cache, block_table, code, None, split_pages,
                     kernel_path, k_scale, v_scale)
    if workspace is None:
        workspace = workspace_for(dims, q_len, n_sink, window, q.device)
    if workspace is not None:
        dims.workspace = ctypes.c_void_p(workspace.data_ptr())
        dims.workspace_bytes = workspace.numel() * workspace.element_size()
    if tree_mask is None:
        st = lib.paged_decode_attention(
            ctypes.byref(dims), q.data_ptr(), k_cache.data_ptr(),
            v_cache.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(),
            int(q_len), int(n_sink), int(window), float(scale),
            out.data_ptr(), lse.data_ptr(), _stream_handle(stream, q.device))
        _check("paged_decode_attention", st)
    else:
        st = lib.paged_tree_attention(
            ctypes.byref(dims), q.data_ptr(), k_cache.data_ptr(),
            v_cache.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(),
            int(q_len), tree_mask.data_ptr(), float(scale), out.data_ptr(),
            lse.data_ptr(), _stream_handle(stream, q.device))
        _check("paged_tree_attention", st)
    return out, lse


def kv_append(k_new, v_new, k_cache, v_cache, block_table, seq_lens,
              stream=None, k_scale=1.0, v_scale=1.0):
    """Scatter k_new/v_new [B, n_new, Hkv, D] into the paged caches in place
    (include/svp.h: kv_append).  seq_lens are the lengths after the append.
    Into FP8 caches the bf16 rows are quantised with k_scale / v_scale."""
    lib = load_library()
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (k_cache, "k_cache"),
                 (v_cache, "v_cache"), (block_table, "block_table"),
                 (seq_lens, "seq_lens")):
        _cuda_contig(t, n)
    code = _cache_code(k_cache, k_new.dtype)
    _need(v_new.dtype == k_new.dtype and v_cache.dtype == k_cache.dtype,
          "k_new/v_new and k_cache/v_cache must pair up")
    B, n_new, Hkv, D = k_new.shape
    dims = make_dims((B, n_new, Hkv, D), k_cache, block_table, code,
                     k_scale=k_scale, v_scale=v_scale)
    st = lib.kv_append(ctypes.byref(dims), k_new.data_ptr(), v_new.data_ptr(),
                       k_cache.data_ptr(), v_cache.data_ptr(),
                       block_table.data_ptr(), seq_lens.data_ptr(), int(n_new),
                       _stream_handle(stream, k_cache.device))
    _check("kv_append", st)


def spec_accept(target_logits, draft_logits, draft_tokens, uniforms,
                out_tokens=None, n_accepted=None, stream=None,
                temperature=1.0, allowed=None, greedy=False):
    """Speculative acceptance (include/svp.h: spec_accept; with a
    temperature other than 1, an `allowed` token mask (int32/uint32
    [B, K+1, ceil(V/32)] on the GPU) or greedy=True: spec_accept_ex).
    Returns (out_tokens [B, K+1] int32, n_accepted [B] int32)."""
    lib = load_library()
    for t, n in ((target_logits, "target_logits"),
                 (draft_logits, "draft_logits"), (draft_tokens, "draft_tokens"),
                 (uniforms, "uniforms")):
        _cuda_contig(t, n)
    _need(target_logits.dtype == torch.float32 and
          draft_logits.dtype == torch.float32 and
          uniforms.dtype == torch.float32, "logits/uniforms must be float32")
    _need(draft_tokens.dtype == torch.int32, "draft_tokens must be int32")
    B, K1, V = target_logits.shape
    K = K1 - 1
    _need(tuple(draft_logits.shape) == (B, K, V), "draft_logits must be [B, K, V]")
    _need(tuple(draft_tokens.shape) == (B, K), "draft_tokens must be [B, K]")
    _need(tuple(uniforms.shape) == (B, K + 1), "uniforms must be [B, K+1]")
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if n_accepted is None:
        n_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    if temperature == 1.0 and allowed is None and not greedy:
        st = lib.spec_accept(B, K, V, target_logits.data_ptr(),
                             draft_logits.data_ptr(), draft_tokens.data_ptr(),
                             uniforms.data_ptr(), out_tokens.data_ptr(),
                             n_accepted.data_ptr(), _stream_handle(stream, dev))
        _check("spec_accept", st)
        return out_tokens, n_accepted
    if allowed is not None:
        _cuda_contig(allowed, "allowed")
        _need(tuple(allowed.shape) == (B, K + 1, (V + 31) // 32) and
              allowed.element_size() == 4,
              "allowed must be 32-bit [B, K+1, ceil(V/32)]")
    opts = SvpAcceptOpts(float(temperature),
                         None if allowed is None else allowed.data_ptr(),
                         int(bool(greedy)))
    st = lib.spec_accept_ex(B, K, V, target_logits.data_ptr(),
                            draft_logits.data_ptr(), draft_tokens.data_ptr(),
                            uniforms.data_ptr(), ctypes.byref(opts),
                            out_tokens.data_ptr(), n_accepted.data_ptr(),
                            _stream_handle(stream, dev))
    _check("spec_accept_ex", st)
    return out_tokens, n_accepted


def spec_accept_tree(target_logits, draft_logits, parents, node_tokens,
                     uniforms, out_tokens=None, out_nodes=None,
                     n_accepted=None, stream=None):
    """Tree acceptance (include/svp.h: spec_accept_tree).  Returns
    (out_tokens [B, N] int32, out_nodes [B, N] int32, n_accepted [B] int32)."""
    lib = load_library()
    for t, n in ((target_logits, "target_logits"),
                 (draft_logits, "draft_logits"), (parents, "parents"),
                 (node_tokens, "node_tokens"), (uniforms, "uniforms")):
        _cuda_contig(t, n)
    _need(target_logits.dtype == torch.float32 and
          draft_logits.dtype == torch.float32 and
          uniforms.dtype == torch.float32, "logits/uniforms must be float32")
    _need(parents.dtype == torch.int32 and node_tokens.dtype == torch.int32,
          "parents/node_tokens must be int32")
    B, N, V = target_logits.shape
    _need(tuple(draft_logits.shape) == (B, N, V), "draft_logits must be [B, N, V]")
    for t, n in ((parents, "parents"), (node_tokens, "node_tokens"),
                 (uniforms, "uniforms")):
        _need(tuple(t.shape) == (B, N), f"{n} must be [B, N]")
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty((B, N), dtype=torch.int32, device=dev)
    if out_nodes is None:
        out_nodes = torch.empty((B, N), dtype=torch.int32, device=dev)
    if n_accepted is None:
        n_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    st = lib.spec_accept_tree(B, N, V, target_logits.data_ptr(),
                              draft_logits.data_ptr(), parents.data_ptr(),
                              node_tokens.data_ptr(), uniforms.data_ptr(),
                              out_tokens.data_ptr(), out_nodes.data_ptr(),
                              n_accepted.data_ptr(), _stream_handle(stream, dev))
    _check("spec_accept_tree", st)
    return out_tokens, out_nodes, n_accepted


def read_device_status(stream=None, device=None) -> int:
    """Synchronise and return (and clear) the device-side SVP_DEV_* flags."""
    lib = load_library()
    flags = ctypes.c_int(0)
    st = lib.svp_read_device_status(_stream_handle(stream, device),
                                    ctypes.byref(flags))
    _check("svp_read_device_status", st)
    return flags.value


def last_launch_count() -> int:
    """Kernels launched by the last successful library call on this thread."""
    return int(load_library().svp_last_launch_count())


class StepRunner:
    """The graph-captured decode step (include/svp.h: svp_step_*): two
    ping-pong slots of pinned host buffers, each replayed as one CUDA graph
    (input copy, kv_append, attention, acceptance) with its result copied
    back on a separate stream.  host(slot, name) returns a numpy view of a
    slot's pinned buffer (bf16 as uint16 bits).  Draft chains take the
    verify epilogue options (temperature, greedy, use_mask: the token mask
    in field "allowed"); tree_nodes > 0 makes the step a draft-tree verify
    (fields "tree_mask", "parents", "node_tokens"; result "out_nodes")."""

    def __init__(self, k_cache, v_cache, batch, num_q_heads, q_len,
                 max_blocks_per_seq, n_sink=0, window=0, scale=None,
                 num_draft=0, vocab=0, split_pages=0, kernel_path=PATH_AUTO,
                 k_scale=1.0, v_scale=1.0, temperature=1.0, greedy=False,
                 use_mask=False, tree_nodes=0):
        lib = load_library()
        _cuda_contig(k_cache, "k_cache")
        _cuda_contig(v_cache, "v_cache")
        nb, Hkv, bs, D = k_cache.shape
        code = (SVP_FP8_E4M3 if k_cache.dtype in _FP8_TYPES
                else _dtype_code(k_cache))
        dims = SvpDims(batch, num_q_heads, Hkv, D, bs, max_blocks_per_seq, nb,
                       code, None, 0, split_pages, kernel_path, k_scale,
                       v_scale)
        if scale is None:
            scale = 1.0 / math.sqrt(D)
        desc = SvpStepDesc(dims, q_len, n_sink, window, float(scale),
                           k_cache.data_ptr(), v_cache.data_ptr(), num_draft,
                           vocab, float(temperature), int(bool(greedy)),
                           int(bool(use_mask)), int(tree_nodes))
        h = ctypes.c_void_p()
        _check("svp_step_create", lib.svp_step_create(ctypes.byref(desc),
                                                      ctypes.byref(h)))
        self._lib, self._h = lib, h
        self._keep = (k_cache, v_cache)
        ed = np.float32 if code == SVP_F32 else np.uint16
        B, Q, K, V, N = batch, q_len, num_draft, vocab, tree_nodes
        rt = N if N else K + 1   # target rows, uniforms, output tokens
        rd = N if N else K       # draft rows
        self._spec = {
            "q": (ed, (B, Q, num_q_heads, D)), "k_new": (ed, (B, Q, Hkv, D)),
            "v_new": (ed, (B, Q, Hkv, D)),
            "block_table": (np.int32, (B, max_blocks_per_seq)),
            "seq_lens": (np.int32, (B,)),
            "target_logits": (np.float32, (B, rt, V)),
            "draft_logits": (np.float32, (B, rd, V)),
            "draft_tokens": (np.int32, (B, K)),
            "uniforms": (np.float32, (B, rt)),
            "out": (ed, (B, Q, num_q_heads, D)),
            "lse": (np.float32, (B, Q, num_q_heads)),
            "out_tokens": (np.int32, (B, rt)),
            "n_accepted": (np.int32, (B,)),
            "allowed": (np.uint32, (B, K + 1, (V + 31) // 32)),
            "tree_mask": (np.uint32, (B, N)),
            "parents": (np.int32, (B, N)),
            "node_tokens": (np.int32, (B, N)),
            "out_nodes": (np.int32, (B, N)),
        }
        self._views = {}

    def host(self, slot, name):
        key = (slot, name)
        if key not in self._views:
            n = ctypes.c_size_t()
            ptr = self._lib.svp_step_host_buffer(self._h, slot,
                                                 STEP_FIELDS.index(name),
                                                 ctypes.byref(n))
            _need(ptr is not None, f"slot {slot} has no field {name}")
            raw = (ctypes.c_uint8 * n.value).from_address(ptr)
            dt, shape = self._spec[name]
            self._views[key] = np.frombuffer(raw, dtype=dt).reshape(shape)
        return self._views[key]

    def launch(self, slot):
        _check("svp_step_launch", self._lib.svp_step_launch(self._h, slot))

    def wait(self, slot):
        _check("svp_step_wait", self._lib.svp_step_wait(self._h, slot))

    def close(self):
        if self._h:
            self._views.clear()
            _check("svp_step_destroy", self._lib.svp_step_destroy(self._h))
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
