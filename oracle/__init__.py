"""fp64 CPU oracle for paged decode/verify attention, KV append and
speculative acceptance.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product package
(``spec_verify_paged_gb300``) never does, and this package never imports it.
The arithmetic lives in ``oracle.c`` (plain single-threaded C, fp64); this
module only builds it with gcc and marshals numpy arrays into it.

Which page passage each function follows is stated in ``oracle.c``:
exact attention from the lesson "KV cache & Flash Attention" (section
"FlashAttention -- the tiling trick") and the StreamingLLM page (section "The
softmax problem"); masks from "How speculative decoding doubles LLM speed"
(step 2, verification) and the StreamingLLM page (section "The StreamingLLM
solution"); acceptance from "How speculative decoding doubles LLM speed"
(step 3, sampling); the draft-tree mask and tree acceptance from the same
page (section "Modern architecture variants", SpecInfer) and "Speculative
decoding: how AI models get faster without getting bigger" (section on
real-world adoption).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1
BOUNDARY_EPS = 1e-6


def build(force: bool = False) -> str:
    """Compile liboracle.so in place with gcc (-O2, no fast-math, no threads)."""
    stale = (not os.path.exists(_LIB)) or any(
        os.path.getmtime(s) > os.path.getmtime(_LIB) for s in (_SRC, _HDR))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
            lib.oracle_paged_attention.argtypes = (
                [i32] * 8 + [vp] * 5 + [i32, i32, i32, f32, vp, i64, vp, vp])
            lib.oracle_paged_attention.restype = i32
            lib.oracle_paged_attention_tiled.argtypes = (
                [i32] * 8 + [vp] * 5 + [i32, i32, i32, f32, i32, i32, vp, vp])
            lib.oracle_paged_attention_tiled.restype = i32
            lib.oracle_kv_append.argtypes = [i32] * 7 + [vp] * 6 + [i32]
            lib.oracle_kv_append.restype = i32
            lib.oracle_spec_accept.argtypes = (
                [i32] * 3 + [vp] * 8 + [ctypes.c_double])
            lib.oracle_spec_accept.restype = i32
            lib.oracle_paged_tree_attention.argtypes = (
                [i32] * 8 + [vp] * 5 + [i32, vp, f32, vp, i64, vp, vp])
            lib.oracle_paged_tree_attention.restype = i32
            lib.oracle_spec_accept_tree.argtypes = (
                [i32] * 3 + [vp] * 10 + [ctypes.c_double])
            lib.oracle_spec_accept_tree.restype = i32
            lib.oracle_spec_accept_ex.argtypes = (
                [i32] * 3 + [vp] * 4 + [ctypes.c_double, vp, i32, vp, vp, vp,
                                        ctypes.c_double])
            lib.oracle_spec_accept_ex.restype = i32
            lib.oracle_spec_accept_valid.argtypes = (
                [i32] * 3 + [vp] * 4 + [ctypes.c_double] + [vp] * 4 +
                [i32, ctypes.c_double])
            lib.oracle_spec_accept_valid.restype = i32
            lib.oracle_spec_accept_tree_valid.argtypes = (
                [i32] * 3 + [vp] * 7 + [i32, i32, ctypes.c_double])
            lib.oracle_spec_accept_tree_valid.restype = i32
            lib.oracle_paged_attention_fp8.argtypes = (
                [i32] * 7 + [vp] * 3 + [ctypes.c_double] * 2 + [vp] * 2 +
                [i32, i32, i32, f32, vp, i64, vp, vp])
            lib.oracle_paged_attention_fp8.restype = i32
            lib.oracle_e4m3_decode.argtypes = [vp, ctypes.c_long, vp]
            lib.oracle_e4m3_decode.restype = i32
            lib.oracle_e4m3_encode.argtypes = [vp, ctypes.c_long, f32, vp]
            lib.oracle_e4m3_encode.restype = i32
            lib.oracle_kv_append_fp8.argtypes = ([i32] * 6 + [vp] * 4 +
                                                 [f32, f32, vp, vp, i32])
            lib.oracle_kv_append_fp8.restype = i32
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(arr):
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.uint16:  # raw bfloat16 bit patterns
        return BF16
    raise TypeError(f"oracle takes float32 or uint16 (bf16 bits), got {arr.dtype}")


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def paged_attention(q, k_cache, v_cache, block_table, seq_lens, q_len,
                    n_sink=0, window=0, scale=None, rows=None, tiled=None):
    """Exact attention over the paged cache, in fp64.

    q: [B, q_len, Hq, D]; k_cache/v_cache: [num_blocks, Hkv, block_size, D]
    (float32 or uint16 bf16 bits, same dtype as q); block_table [B, max_blocks]
    int32; seq_lens [B] int32 (including the q_len new rows).
    rows: optional flat row ids (b*q_len + i)*Hq + h; then returns
    (out [n, D], lse [n]).  Otherwise returns out [B, q_len, Hq, D] and
    lse [B, q_len, Hq] (float64).
    tiled=(tile, n_splits) runs the tiled/split online-softmax variant.
    """
    lib = _load()
    B, ql, Hq, D = q.shape
    assert ql == q_len
    nb, Hkv, bs, D2 = k_cache.shape
    assert D2 == D and v_cache.shape == k_cache.shape
    code = _dtype_code(q)
    assert _dtype_code(k_cache) == code and _dtype_code(v_cache) == code
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    q = _c(q, q.dtype)
    kc = _c(k_cache, k_cache.dtype)
    vc = _c(v_cache, v_cache.dtype)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    mb = bt.shape[1] if bt.ndim == 2 else 0
    if tiled is not None:
        out = np.zeros((B, q_len, Hq, D), np.float64)
        lse = np.zeros((B, q_len, Hq), np.float64)
        st = lib.oracle_paged_attention_tiled(
            B, Hq, Hkv, D, bs, mb, nb, code, _ptr(q), _ptr(kc), _ptr(vc),
            _ptr(bt), _ptr(sl), q_len, n_sink, window, float(scale),
            int(tiled[0]), int(tiled[1]), _ptr(out), _ptr(lse))
    elif rows is None:
        out = np.zeros((B, q_len, Hq, D), np.float64)
        lse = np.zeros((B, q_len, Hq), np.float64)
        st = lib.oracle_paged_attention(
            B, Hq, Hkv, D, bs, mb, nb, code, _ptr(q), _ptr(kc), _ptr(vc),
            _ptr(bt), _ptr(sl), q_len, n_sink, window, float(scale), None, 0,
            _ptr(out), _ptr(lse))
    else:
        r = _c(rows, np.int64)
        out = np.zeros((r.size, D), np.float64)
        lse = np.zeros((r.size,), np.float64)
        st = lib.oracle_paged_attention(
            B, Hq, Hkv, D, bs, mb, nb, code, _ptr(q), _ptr(kc), _ptr(vc),
            _ptr(bt), _ptr(sl), q_len, n_sink, window, float(scale), _ptr(r),
            r.size, _ptr(out), _ptr(lse))
    if st != 0:
        raise ValueError(f"oracle_paged_attention failed with status {st}")
    return out, lse


def kv_append(k_new, v_new, k_cache, v_cache, block_table, seq_lens):
    """Scatter k_new/v_new [B, n_new, Hkv, D] into copies of the caches.
    Returns the updated (k_cache, v_cache); the inputs are not modified."""
    lib = _load()
    B, n_new, Hkv, D = k_new.shape
    nb, Hkv2, bs, D2 = k_cache.shape
    assert Hkv2 == Hkv and D2 == D and k_new.dtype == k_cache.dtype
    kc = np.array(k_cache, copy=True, order="C")
    vc = np.array(v_cache, copy=True, order="C")
    kn = _c(k_new, k_new.dtype)
    vn = _c(v_new, v_new.dtype)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    st = lib.oracle_kv_append(B, Hkv, D, bs, bt.shape[1], nb, kc.itemsize,
                              _ptr(kn), _ptr(vn), _ptr(kc), _ptr(vc), _ptr(bt),
                              _ptr(sl), n_new)
    if st != 0:
        raise ValueError(f"oracle_kv_append failed with status {st}")
    return kc, vc


def spec_accept(target_logits, draft_logits, draft_tokens, uniforms,
                eps=BOUNDARY_EPS):
    """Literal rejection-sampling loop in fp64.

    Returns dict(out_tokens [B, K+1] int32 (-1 padded), n_accepted [B] int32,
    near_boundary [B] int32, residual_fallback [B] int32)."""
    lib = _load()
    B, K1, V = target_logits.shape
    K = K1 - 1
    assert draft_logits.shape == (B, K, V)
    assert draft_tokens.shape == (B, K) and uniforms.shape == (B, K + 1)
    tl = _c(target_logits, np.float32)
    dl = _c(draft_logits, np.float32)
    dt = _c(draft_tokens, np.int32)
    un = _c(uniforms, np.float32)
    out = np.full((B, K + 1), -1, np.int32)
    nacc = np.zeros((B,), np.int32)
    near = np.zeros((B,), np.int32)
    fb = np.zeros((B,), np.int32)
    st = lib.oracle_spec_accept(B, K, V, _ptr(tl), _ptr(dl), _ptr(dt), _ptr(un),
                                _ptr(out), _ptr(nacc), _ptr(near), _ptr(fb),
                                float(eps))
    if st != 0:
        raise ValueError(f"oracle_spec_accept failed with status {st}")
    return {"out_tokens": out, "n_accepted": nacc, "near_boundary": near,
            "residual_fallback": fb}


def paged_tree_attention(q, k_cache, v_cache, block_table, seq_lens, q_len,
                         tree_mask, scale=None, rows=None):
    """Exact attention with a draft-tree mask, in fp64.

    tree_mask [B, q_len] uint32: bit k of entry (b, i) set iff node k is an
    ancestor of node i or i itself (keys of the q_len new rows); every key
    before them is visible.  Returns like paged_attention."""
    lib = _load()
    B, ql, Hq, D = q.shape
    assert ql == q_len and tree_mask.shape == (B, q_len)
    nb, Hkv, bs, D2 = k_cache.shape
    assert D2 == D and v_cache.shape == k_cache.shape
    code = _dtype_code(q)
    assert _dtype_code(k_cache) == code and _dtype_code(v_cache) == code
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    q = _c(q, q.dtype)
    kc = _c(k_cache, k_cache.dtype)
    vc = _c(v_cache, v_cache.dtype)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    tm = _c(tree_mask, np.uint32)
    mb = bt.shape[1] if bt.ndim == 2 else 0
    if rows is None:
        out = np.zeros((B, q_len, Hq, D), np.float64)
        lse = np.zeros((B, q_len, Hq), np.float64)
        r, n = None, 0
    else:
        r = _c(rows, np.int64)
        out = np.zeros((r.size, D), np.float64)
        lse = np.zeros((r.size,), np.float64)
        n = r.size
    st = lib.oracle_paged_tree_attention(
        B, Hq, Hkv, D, bs, mb, nb, code, _ptr(q), _ptr(kc), _ptr(vc),
        _ptr(bt), _ptr(sl), q_len, _ptr(tm), float(scale), _ptr(r), n,
        _ptr(out), _ptr(lse))
    if st != 0:
        raise ValueError(f"oracle_paged_tree_attention failed with status {st}")
    return out, lse


def spec_accept_tree(target_logits, draft_logits, parents, node_tokens,
                     uniforms, eps=BOUNDARY_EPS):
    """Literal tree walk in fp64 (see oracle.h).

    target_logits, draft_logits [B, N, V] fp32; parents, node_tokens [B, N]
    int32; uniforms [B, N] fp32.  Returns dict(out_tokens [B, N],
    out_nodes [B, N], n_accepted [B], near_boundary [B],
    residual_fallback [B])."""
    lib = _load()
    B, N, V = target_logits.shape
    assert draft_logits.shape == (B, N, V)
    assert parents.shape == (B, N) and node_tokens.shape == (B, N)
    assert uniforms.shape == (B, N)
    tl = _c(target_logits, np.float32)
    dl = _c(draft_logits, np.float32)
    pa = _c(parents, np.int32)
    tk = _c(node_tokens, np.int32)
    un = _c(uniforms, np.float32)
    out = np.full((B, N), -1, np.int32)
    nodes = np.full((B, N), -1, np.int32)
    nacc = np.zeros((B,), np.int32)
    near = np.zeros((B,), np.int32)
    fb = np.zeros((B,), np.int32)
    st = lib.oracle_spec_accept_tree(B, N, V, _ptr(tl), _ptr(dl), _ptr(pa),
                                     _ptr(tk), _ptr(un), _ptr(out), _ptr(nodes),
                                     _ptr(nacc), _ptr(near), _ptr(fb),
                                     float(eps))
    if st != 0:
        raise ValueError(f"oracle_spec_accept_tree failed with status {st}")
    return {"out_tokens": out, "out_nodes": nodes, "n_accepted": nacc,
            "near_boundary": near, "residual_fallback": fb}


def spec_accept_ex(target_logits, draft_logits, draft_tokens, uniforms,
                   temperature=1.0, allowed=None, greedy=False,
                   eps=BOUNDARY_EPS):
    """spec_accept with the verify epilogue (see oracle.h): temperature,
    allowed [B, K+1, ceil(V/32)] uint32 token masks (or None), greedy.
    Returns dict(out_tokens, n_accepted, near_boundary)."""
    lib = _load()
    B, K1, V = target_logits.shape
    K = K1 - 1
    assert draft_logits.shape == (B, K, V)
    assert draft_tokens.shape == (B, K) and uniforms.shape == (B, K + 1)
    tl = _c(target_logits, np.float32)
    dl = _c(draft_logits, np.float32)
    dt = _c(draft_tokens, np.int32)
    un = _c(uniforms, np.float32)
    al = None
    if allowed is not None:
        al = _c(allowed, np.uint32)
        assert al.shape == (B, K + 1, (V + 31) // 32)
    out = np.full((B, K + 1), -1, np.int32)
    nacc = np.zeros((B,), np.int32)
    near = np.zeros((B,), np.int32)
    st = lib.oracle_spec_accept_ex(B, K, V, _ptr(tl), _ptr(dl), _ptr(dt),
                                   _ptr(un), float(temperature), _ptr(al),
                                   int(bool(greedy)), _ptr(out), _ptr(nacc),
                                   _ptr(near), float(eps))
    if st != 0:
        raise ValueError(f"oracle_spec_accept_ex failed with status {st}")
    return {"out_tokens": out, "n_accepted": nacc, "near_boundary": near}


MAX_CAND = 16


def spec_accept_valid(target_logits, draft_logits, draft_tokens, uniforms,
                      temperature=1.0, allowed=None, eps=BOUNDARY_EPS,
                      max_cand=MAX_CAND):
    """The outcomes the linear rule can reach when every comparison within
    eps of its boundary may go either way (see oracle.h).

    Returns dict(path_valid [B, K+1] bool: entry j < K = "first rejection at
    j", entry K = "all accepted"; cand [B, K+1, max_cand] int32 (-1 padded);
    n_cand [B, K+1])."""
    lib = _load()
    B, K1, V = target_logits.shape
    K = K1 - 1
    assert draft_logits.shape == (B, K, V)
    assert draft_tokens.shape == (B, K) and uniforms.shape == (B, K + 1)
    tl = _c(target_logits, np.float32)
    dl = _c(draft_logits, np.float32)
    dt = _c(draft_tokens, np.int32)
    un = _c(uniforms, np.float32)
    al = None
    if allowed is not None:
        al = _c(allowed, np.uint32)
        assert al.shape == (B, K + 1, (V + 31) // 32)
    pv = np.zeros((B, K + 1), np.int32)
    cand = np.full((B, K + 1, max_cand), -1, np.int32)
    ncand = np.zeros((B, K + 1), np.int32)
    st = lib.oracle_spec_accept_valid(B, K, V, _ptr(tl), _ptr(dl), _ptr(dt),
                                      _ptr(un), float(temperature), _ptr(al),
                                      _ptr(pv), _ptr(cand), _ptr(ncand),
                                      int(max_cand), float(eps))
    if st != 0:
        raise ValueError(f"oracle_spec_accept_valid failed with status {st}")
    return {"path_valid": pv.astype(bool), "cand": cand, "n_cand": ncand}


def spec_accept_tree_valid(target_logits, draft_logits, parents, node_tokens,
                           uniforms, eps=BOUNDARY_EPS, max_out=64,
                           max_cand=MAX_CAND):
    """The outcomes the tree walk can reach when every comparison within eps
    of its boundary may go either way (see oracle.h).

    Returns a list (one per sequence) of outcomes, each a dict(nodes: tuple
    of accepted nodes, n_accepted, cand: tuple of candidate tokens of the
    final draw, n_cand)."""
    lib = _load()
    B, N, V = target_logits.shape
    assert draft_logits.shape == (B, N, V)
    assert parents.shape == (B, N) and node_tokens.shape == (B, N)
    assert uniforms.shape == (B, N)
    tl = _c(target_logits, np.float32)
    dl = _c(draft_logits, np.float32)
    pa = _c(parents, np.int32)
    tk = _c(node_tokens, np.int32)
    un = _c(uniforms, np.float32)
    stride = N + 2 + max_cand
    rows = np.full((B, max_out, stride), -1, np.int32)
    nout = np.zeros((B,), np.int32)
    st = lib.oracle_spec_accept_tree_valid(B, N, V, _ptr(tl), _ptr(dl),
                                           _ptr(pa), _ptr(tk), _ptr(un),
                                           _ptr(rows), _ptr(nout),
                                           int(max_out), int(max_cand),
                                           float(eps))
    if st != 0:
        raise ValueError(f"oracle_spec_accept_tree_valid failed with status {st}")
    res = []
    for b in range(B):
        outs = []
        for o in range(min(int(nout[b]), max_out)):
            r = rows[b, o]
            n = int(r[N])
            nc = int(r[N + 1])
            outs.append({"nodes": tuple(int(v) for v in r[:n]),
                         "n_accepted": n, "n_cand": nc,
                         "cand": tuple(int(v) for v in r[N + 2:N + 2 + min(nc, max_cand)])})
        res.append({"outcomes": outs, "n_outcomes": int(nout[b])})
    return res


def e4m3_decode(codes):
    """Values of FP8 E4M3 codes (uint8 array) as float64."""
    lib = _load()
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    lib.oracle_e4m3_decode(_ptr(c), c.size, _ptr(out))
    return out


def e4m3_encode(x, scale=1.0):
    """E4M3 codes of float32 x / scale (nearest, ties to even, saturating)."""
    lib = _load()
    a = _c(x, np.float32)
    out = np.empty(a.shape, np.uint8)
    if lib.oracle_e4m3_encode(_ptr(a), a.size, float(scale), _ptr(out)) != 0:
        raise ValueError("scale must be positive")
    return out


def paged_attention_fp8(q, k_cache, v_cache, k_scale, v_scale, block_table,
                        seq_lens, q_len, n_sink=0, window=0, scale=None,
                        rows=None):
    """Exact attention over FP8 E4M3 caches (uint8 codes; values scaled by
    k_scale / v_scale) with bf16 q (uint16 bits), in fp64."""
    lib = _load()
    B, ql, Hq, D = q.shape
    assert ql == q_len and q.dtype == np.uint16
    nb, Hkv, bs, D2 = k_cache.shape
    assert D2 == D and k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    q = _c(q, np.uint16)
    kc = _c(k_cache, np.uint8)
    vc = _c(v_cache, np.uint8)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    if rows is None:
        out = np.zeros((B, q_len, Hq, D), np.float64)
        lse = np.zeros((B, q_len, Hq), np.float64)
        r, n = None, 0
    else:
        r = _c(rows, np.int64)
        out = np.zeros((r.size, D), np.float64)
        lse = np.zeros((r.size,), np.float64)
        n = r.size
    st = lib.oracle_paged_attention_fp8(
        B, Hq, Hkv, D, bs, bt.shape[1], nb, _ptr(q), _ptr(kc), _ptr(vc),
        float(k_scale), float(v_scale), _ptr(bt), _ptr(sl), q_len, n_sink,
        window, float(scale), _ptr(r), n, _ptr(out), _ptr(lse))
    if st != 0:
        raise ValueError(f"oracle_paged_attention_fp8 failed with status {st}")
    return out, lse


def kv_append_fp8(k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                  block_table, seq_lens):
    """Quantise bf16 k_new / v_new into copies of FP8 caches."""
    lib = _load()
    B, n_new, Hkv, D = k_new.shape
    nb, Hkv2, bs, D2 = k_cache.shape
    assert Hkv2 == Hkv and D2 == D and k_cache.dtype == np.uint8
    kc = np.array(k_cache, copy=True, order="C")
    vc = np.array(v_cache, copy=True, order="C")
    kn = _c(k_new, np.uint16)
    vn = _c(v_new, np.uint16)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    st = lib.oracle_kv_append_fp8(B, Hkv, D, bs, bt.shape[1], nb, _ptr(kn),
                                  _ptr(vn), _ptr(kc), _ptr(vc), float(k_scale),
                                  float(v_scale), _ptr(bt), _ptr(sl), n_new)
    if st != 0:
        raise ValueError(f"oracle_kv_append_fp8 failed with status {st}")
    return kc, vc
