"""Benchmark: paged decode attention step on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--split-pages P] [--kernel-path 0-3]
                    [--no-graph]

A step is one pass of the hot path over one batch: kv_append of the
batch's new K/V rows into the paged cache, then paged_decode_attention of
the new query rows over every cached row (decode-7b: 32 sequences, 32/32
heads, head_dim 128, context U[512, 4096], bf16 16-token pages in a shuffled
block table); on the verify workloads (q_len > 1) the step ends with
spec_accept of the q_len - 1 drafts per sequence over a 32,000-token
vocabulary (its time is reported as `accept_us`); the tree-verify workload
(a 15-node binary draft tree per sequence) runs paged_tree_attention and
spec_accept_tree instead.  After the warm-up the
step is captured as CUDA graphs and the timed loop replays them, so the
host's launch overhead does not pace the GPU.  `value` is query tokens per
second over the whole job; the KV-read bandwidth of the attention call and
its fraction of the measured HBM peak are in `roofline`.  Inputs are
resident in HBM before the timed region; each step reads 0.27-2.2 GB of
KV, more than the 129 MB L2, so no flush is needed.  `e2e` repeats the
step through the plain public calls with the step's inputs copied from
pinned host memory and its outputs copied back inside the timed region.
`cpu_baseline` times the fp64 CPU oracle on a bounded sample.

--impl reference times that CPU oracle alone (the slow, obviously correct
program the GPU results are checked against) on the same workload.

Multi-GPU: one process per GPU under torchrun; each rank runs an
independent replica of the workload (the path shards by sequence with no
exchange), timing is the max over ranks, value is the sum of the work.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from spec_verify_paged_gb300 import accounting as A  # noqa: E402
from spec_verify_paged_gb300 import workloads as W  # noqa: E402

METRIC = ("decode-attention query-tokens/s and achieved KV-read HBM GB/s "
          "(% of GB300 peak)")
UNIT = "query-tokens/s"
CSRC = os.path.join(ROOT, "spec_verify_paged_gb300", "csrc")


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def attention_kernel(cfg, kernel_path):
    """(kernel name, its source file) for the path the library takes: the
    tcgen05 kernel for bf16 head_dim-128 groups of 3+ query rows, the
    CUDA-core / mma.sync kernel otherwise."""
    rows = cfg.q_len * (cfg.num_q_heads // cfg.num_kv_heads)
    tc = (kernel_path == 3 or
          (kernel_path == 0 and cfg.dtype == "bf16" and cfg.head_dim == 128
           and rows >= 3))
    if tc:
        return "paged_attention_tc_kernel", "attention_tc.cu"
    return "paged_attention_kernel", "attention.cu"


def code_hash(path):
    """sha256 prefix of a source's code: `//` comments and blank lines
    removed, so an edit of comments alone leaves it unchanged."""
    lines = []
    for line in open(path, encoding="utf-8"):
        code = line.split("//", 1)[0].rstrip()
        if code:
            lines.append(code)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def kernel_traffic(kernel, src, workload):
    """dram bytes per launch from the committed ncu summary of this kernel
    on this workload, if it was taken on the current code; else None."""
    prof = os.path.join(ROOT, "profiles", f"ncu_{kernel}_{workload}.md")
    if not os.path.exists(prof):
        return None
    sha = code_hash(os.path.join(CSRC, src))
    vals = {}
    for line in open(prof):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            quoted = re.findall(r"`([^`]*)`", v)
            vals[k.strip()] = quoted[0] if quoted else v.strip()
    if vals.get(f"{src} code sha256 prefix") != sha:
        return None
    try:
        return int(vals["dram bytes per launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self._thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self._thread = threading.Thread(target=self._read, daemon=True)
        self._thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=2)

    def summary(self, t0, t1):
        rows = [s for t, s in self.samples if t0 - 0.06 <= t <= t1 + 0.06]
        if not rows:  # a very short region: the nearest samples around it
            near = sorted(self.samples, key=lambda ts: abs(ts[0] - (t0 + t1) / 2))
            rows = [s for _, s in near[:3]]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def to_dev(a, dev):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def to_pinned(a):
    import torch
    if a.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    return t.pin_memory()


def pack_buffers(parts, dev):
    """One pinned host buffer and one device buffer holding the given
    tensors back to back (256-byte aligned); returns (host, device, views of
    the device buffer shaped like the parts)."""
    import torch
    offs, total = [], 0
    for _, t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    devb = torch.empty(total, dtype=torch.uint8, device=dev)
    views = {}
    for (name, t), o in zip(parts, offs):
        n = t.numel() * t.element_size()
        views[name] = devb[o:o + n].view(t.dtype).view(t.shape)
    views["_offsets"] = dict(zip([n for n, _ in parts], offs))
    views["_host"] = host
    return host, devb, views


def host_view(host, dview):
    """The host-buffer slice that mirrors a device view from pack_buffers."""
    base = dview.untyped_storage().data_ptr()
    off = dview.data_ptr() - base
    n = dview.numel() * dview.element_size()
    return host[off:off + n].view(dview.dtype).view(dview.shape)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, world: int) -> float:
    """The slowest rank's time (all ranks must call this)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and --impl reference)
# --------------------------------------------------------------------------

def oracle_sample(wl, n_seqs, start=0):
    """Run the fp64 oracle on n_seqs sequences of the workload (all heads,
    all query rows); returns (seconds, query tokens)."""
    import oracle
    oracle.build()
    B = wl.cfg.batch
    per = wl.q_len * wl.cfg.num_q_heads
    seqs = [(start + i) % B for i in range(n_seqs)]
    rows = np.concatenate([np.arange(b * per, (b + 1) * per) for b in seqs])
    t = time.perf_counter()
    if wl.cfg.dtype == "fp8":
        oracle.paged_attention_fp8(wl.q, wl.k_cache, wl.v_cache, wl.k_scale,
                                   wl.v_scale, wl.block_table, wl.seq_lens,
                                   wl.q_len, wl.cfg.n_sink, wl.cfg.window,
                                   wl.scale, rows=rows.astype(np.int64))
    elif wl.tree_mask is not None:
        oracle.paged_tree_attention(wl.q, wl.k_cache, wl.v_cache,
                                    wl.block_table, wl.seq_lens, wl.q_len,
                                    wl.tree_mask, wl.scale,
                                    rows=rows.astype(np.int64))
    else:
        oracle.paged_attention(wl.q, wl.k_cache, wl.v_cache, wl.block_table,
                               wl.seq_lens, wl.q_len, wl.cfg.n_sink,
                               wl.cfg.window, wl.scale,
                               rows=rows.astype(np.int64))
    return time.perf_counter() - t, n_seqs * wl.q_len


def cpu_baseline(wl, budget_s=10.0, max_passes=20):
    """The oracle as it stands, single-threaded, on whole sequences of the
    workload (cycling through them) until about budget_s seconds of CPU
    work."""
    total_t, total_tok, n = 0.0, 0, 0
    while total_t < budget_s and n < max_passes * wl.cfg.batch:
        dt, tok = oracle_sample(wl, 1, start=n)
        total_t += dt
        total_tok += tok
        n += 1
    return {"value": total_tok / total_t, "unit": UNIT, "cores": 1,
            "host_cpus": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{n} sequence passes over the {wl.cfg.batch} sequences "
                      f"of {wl.cfg.name} (all {wl.cfg.num_q_heads} heads, "
                      f"fp64, one thread), {total_t:.1f} s"}


def tokens_per_step_of(cfg):
    return cfg.batch * cfg.q_len


def workload_config(wl, split_pages=None):
    cfg = wl.cfg
    tr = A.attention_traffic(wl.seq_lens, cfg.q_len, cfg.num_q_heads,
                             cfg.num_kv_heads, cfg.head_dim,
                             {"f32": 4, "bf16": 2, "fp8": 1}[cfg.dtype],
                             cfg.n_sink,
                             cfg.window)
    c = {"workload": cfg.name, "batch": cfg.batch,
         "num_q_heads": cfg.num_q_heads, "num_kv_heads": cfg.num_kv_heads,
         "head_dim": cfg.head_dim, "q_len": cfg.q_len, "kv_dtype": cfg.dtype,
         "page_tokens": W.BLOCK_SIZE,
         "context": (f"U[{cfg.ctx_min},{cfg.ctx_max}]"
                     if cfg.ctx_min != cfg.ctx_max else cfg.ctx_min),
         "n_sink": cfg.n_sink, "window": cfg.window,
         "kv_bytes_per_step": tr["kv_bytes"], "seed": cfg.seed,
         "l2": "no flush: each step reads %.2f GB of KV, > 129 MB L2"
               % (tr["kv_bytes"] / 1e9)}
    if cfg.tree_depth > 0:
        c["draft_tree"] = {"shape": "complete binary", "depth": cfg.tree_depth,
                           "nodes": cfg.q_len}
    if split_pages is not None:
        c["split_pages"] = split_pages
    return c, tr


# --------------------------------------------------------------------------
# the GPU arm
# --------------------------------------------------------------------------

def run_ours(args):
    import torch
    import torch.distributed as dist

    import spec_verify_paged_gb300 as svp
    from spec_verify_paged_gb300 import build as svp_build

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        svp_build.build()
    if world > 1:
        dist.barrier()
    svp.load_library()

    cfg = W.CONFIGS[args.workload]
    if args.batch:
        cfg = dataclasses.replace(cfg, batch=args.batch)
    wl = W.make_attention(cfg, n_new=cfg.q_len, poison=False)
    conf, tr = workload_config(wl, args.split_pages or None)
    if args.kernel_path:
        conf["kernel_path"] = {1: "cuda_cores", 2: "tensor_cores",
                               3: "tcgen05"}[args.kernel_path]
    conf["timing"] = ("plain calls" if args.no_graph else
                      "one CUDA graph per step (append, attention, acceptance "
                      "as programmatic dependent launches); phase times from a "
                      "second timed loop of per-phase graphs")

    q = to_dev(wl.q, dev)
    kc, vc = to_dev(wl.k_cache, dev), to_dev(wl.v_cache, dev)
    bt, sl = to_dev(wl.block_table, dev), to_dev(wl.seq_lens, dev)
    kn, vn = to_dev(wl.k_new, dev), to_dev(wl.v_new, dev)
    out = torch.empty_like(q)
    lse = torch.empty((cfg.batch, cfg.q_len, cfg.num_q_heads),
                      dtype=torch.float32, device=dev)
    # verify workloads (q_len > 1) end with the acceptance step on K =
    # q_len - 1 drafts per sequence, vocab 32,000 (the acceptance workload's
    # recipe, same seed as the attention inputs); a draft tree ends with the
    # tree acceptance over its nodes
    tree = cfg.tree_depth > 0
    tm = to_dev(wl.tree_mask.view(np.int32), dev) if tree else None
    acc = None
    acc_opts = {}
    if tree:
        awl = W.make_tree_accept(batch=cfg.batch, depth=cfg.tree_depth,
                                 vocab=W.TREE_ACCEPT_CONFIG["vocab"],
                                 seed=cfg.seed)
        acc_in = [to_dev(x, dev) for x in (awl.target_logits, awl.draft_logits,
                                           awl.parents, awl.node_tokens,
                                           awl.uniforms)]
        acc_out = tuple(torch.empty(shape, dtype=torch.int32, device=dev)
                        for shape in ((cfg.batch, cfg.q_len),
                                      (cfg.batch, cfg.q_len), (cfg.batch,)))
        acc = (acc_in, acc_out)
        conf["accept"] = {"batch": cfg.batch, "tree_nodes": cfg.q_len,
                          "vocab": W.TREE_ACCEPT_CONFIG["vocab"]}
    elif cfg.q_len > 1:
        awl = W.make_accept(batch=cfg.batch, num_draft=cfg.q_len - 1,
                            vocab=W.ACCEPT_CONFIG["vocab"], seed=cfg.seed)
        acc_in = [to_dev(x, dev) for x in (awl.target_logits, awl.draft_logits,
                                           awl.draft_tokens, awl.uniforms)]
        acc_out = (torch.empty((cfg.batch, cfg.q_len), dtype=torch.int32,
                               device=dev),
                   torch.empty((cfg.batch,), dtype=torch.int32, device=dev))
        acc = (acc_in, acc_out)
        conf["accept"] = {"batch": cfg.batch, "num_draft": cfg.q_len - 1,
                          "vocab": W.ACCEPT_CONFIG["vocab"]}
        # the verify epilogue: temperature, token mask, greedy
        acc_opts = {}
        if args.temperature != 1.0:
            acc_opts["temperature"] = args.temperature
        if args.greedy:
            acc_opts["greedy"] = True
        if args.allowed_density > 0:
            V = W.ACCEPT_CONFIG["vocab"]
            mrng = np.random.default_rng(cfg.seed + 7)
            allowed = mrng.random((cfg.batch, cfg.q_len, V)) < args.allowed_density
            allowed[..., 0] = True
            words = (V + 31) // 32
            pad = np.zeros((cfg.batch, cfg.q_len, words * 32), bool)
            pad[..., :V] = allowed
            bits = np.packbits(pad, axis=-1, bitorder="little").view(np.int32)
            acc_opts["allowed"] = to_dev(np.ascontiguousarray(bits), dev)
        if acc_opts:
            conf["accept"]["epilogue"] = {
                "temperature": args.temperature, "greedy": bool(args.greedy),
                "allowed_density": args.allowed_density}
    stream = torch.cuda.current_stream(dev)
    scale = float(wl.scale)
    launches = [0]

    # an FP8 cache's scales (1 otherwise)
    kv_scales = dict(k_scale=wl.k_scale, v_scale=wl.v_scale)

    def attn_call(q_, bt_, sl_, out_, lse_, tm_=None):
        if tree:
            svp.paged_tree_attention(q_, kc, vc, bt_, sl_, tm_, scale=scale,
                                     out=out_, lse=lse_,
                                     split_pages=args.split_pages,
                                     kernel_path=args.kernel_path, **kv_scales)
        else:
            svp.paged_decode_attention(
                q_, kc, vc, bt_, sl_, q_len=cfg.q_len, n_sink=cfg.n_sink,
                window=cfg.window, scale=scale, out=out_, lse=lse_,
                split_pages=args.split_pages, kernel_path=args.kernel_path,
                **kv_scales)

    def accept_with(inputs, outputs, opts=None):
        opts = acc_opts if opts is None else opts
        if tree:
            svp.spec_accept_tree(*inputs, out_tokens=outputs[0],
                                 out_nodes=outputs[1], n_accepted=outputs[2])
        else:
            svp.spec_accept(*inputs, out_tokens=outputs[0],
                            n_accepted=outputs[1], **opts)

    def accept_call():
        accept_with(acc[0], acc[1])
        return svp.last_launch_count()

    def step(ev=None):
        svp.kv_append(kn, vn, kc, vc, bt, sl, **kv_scales)
        n = svp.last_launch_count()
        if ev is not None:
            ev[0].record(stream)
        attn_call(q, bt, sl, out, lse, tm)
        n += svp.last_launch_count()
        if ev is not None:
            ev[1].record(stream)
        if acc is not None:
            n += accept_call()
            if ev is not None:
                ev[2].record(stream)
        launches[0] += n

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    assert svp.read_device_status() == 0, "device status flags raised"

    # The timed loop replays the step as one CUDA graph captured once here
    # (KV append, attention, acceptance: the library launches each kernel as
    # a programmatic dependent of the one before, so inside one graph each
    # launch overlaps the previous kernel's tail): a step of tens of
    # microseconds would otherwise be paced by the host's Python and launch
    # overhead, not by the GPU.  The library keeps no per-call state, so a
    # replay does exactly the work of a call.  The phase times (attention
    # call, acceptance call) come from a second timed loop that replays each
    # phase as its own graph with CUDA events between them.  The end-to-end
    # figure below still goes through the plain public calls every step.
    g_step = None
    if not args.no_graph:
        g_step, g_app, g_attn, g_acc = (torch.cuda.CUDAGraph(),
                                        torch.cuda.CUDAGraph(),
                                        torch.cuda.CUDAGraph(),
                                        torch.cuda.CUDAGraph())
        with torch.cuda.graph(g_app):
            svp.kv_append(kn, vn, kc, vc, bt, sl, **kv_scales)
        n_app = svp.last_launch_count()
        with torch.cuda.graph(g_attn):
            attn_call(q, bt, sl, out, lse, tm)
        n_attn = svp.last_launch_count()
        n_acc = 0
        if acc is not None:
            with torch.cuda.graph(g_acc):
                n_acc = accept_call()
        with torch.cuda.graph(g_step):
            svp.kv_append(kn, vn, kc, vc, bt, sl, **kv_scales)
            attn_call(q, bt, sl, out, lse, tm)
            if acc is not None:
                accept_call()
        torch.cuda.synchronize(dev)

        def whole_step():
            g_step.replay()
            launches[0] += n_app + n_attn + n_acc

        def step(ev=None):  # noqa: F811 -- the replayed form of the step
            g_app.replay()
            if ev is not None:
                ev[0].record(stream)
            g_attn.replay()
            if ev is not None:
                ev[1].record(stream)
            if acc is not None:
                g_acc.replay()
                if ev is not None:
                    ev[2].record(stream)
            launches[0] += n_app + n_attn + n_acc

        for _ in range(3):
            step()
            whole_step()
        torch.cuda.synchronize(dev)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)  # let the sampler start producing lines
    attn_ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3))
               for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches[0] = 0
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        if g_step is not None:
            whole_step()
        else:
            step(attn_ev[i])
    end.record(stream)
    if g_step is not None:  # the phase times, in a second timed loop
        for i in range(args.steps):
            step(attn_ev[i])
    torch.cuda.synchronize(dev)
    t1 = time.time()
    if world > 1:
        dist.barrier()
    gpu_launches = launches[0]
    ms = start.elapsed_time(end)
    attn_ms = [e[0].elapsed_time(e[1]) for e in attn_ev]
    acc_ms = ([e[1].elapsed_time(e[2]) for e in attn_ev] if acc is not None
              else None)
    time.sleep(0.1)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    ms_max = max_over_ranks(ms, world)

    # ---- end to end through the public calls, host buffers ----
    # The step's inputs (q, new K/V rows, block table, lengths) travel in one
    # pinned buffer and one host-to-device copy; out and lse come back in
    # one device-to-host copy that the host waits for every step.
    in_parts = [("q", q), ("k_new", kn), ("v_new", vn), ("block_table", bt),
                ("seq_lens", sl)]
    if tree:
        in_parts.append(("tree_mask", tm))
    acc_names = (("target_logits", "draft_logits", "parents", "node_tokens",
                  "uniforms") if tree else
                 ("target_logits", "draft_logits", "draft_tokens", "uniforms"))
    if acc is not None:
        in_parts += list(zip(acc_names, acc[0]))
    if "allowed" in acc_opts:  # a grammar mask arrives with every step
        in_parts.append(("allowed", acc_opts["allowed"]))
    h_in, d_in, d_views = pack_buffers(in_parts, dev)
    for name, t in in_parts:
        host_view(h_in, d_views[name]).copy_(t.cpu())
    out_parts = [("out", out), ("lse", lse)]
    res_names = (("out_tokens", "out_nodes", "n_accepted") if tree else
                 ("out_tokens", "n_accepted"))
    if acc is not None:
        out_parts += list(zip(res_names, acc[1]))
    h_res, d_res, r_views = pack_buffers(out_parts, dev)

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        svp.kv_append(d_views["k_new"], d_views["v_new"], kc, vc,
                      d_views["block_table"], d_views["seq_lens"], **kv_scales)
        attn_call(d_views["q"], d_views["block_table"], d_views["seq_lens"],
                  r_views["out"], r_views["lse"], d_views.get("tree_mask"))
        if acc is not None:
            e2e_opts = dict(acc_opts)
            if "allowed" in e2e_opts:
                e2e_opts["allowed"] = d_views["allowed"]
            accept_with([d_views[k] for k in acc_names],
                        [r_views[k] for k in res_names], e2e_opts)
        h_res.copy_(d_res, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize(dev)
    e_steps = max(1, min(args.steps, 200))
    if world > 1:
        dist.barrier()
    e0 = time.perf_counter()
    for _ in range(e_steps):
        e2e_step()
        stream.synchronize()           # the host reads the result every step
    e_ms = (time.perf_counter() - e0) * 1e3 / e_steps
    e_ms = max_over_ranks(e_ms, world)
    h2d = sum(t.numel() * t.element_size() for _, t in in_parts)
    d2h = sum(t.numel() * t.element_size() for _, t in out_parts)

    # ---- end to end through the graph-captured step (svp_step_*) ----
    # Two ping-pong slots of pinned buffers; each launch replays the slot's
    # graph (input copy, kv_append, attention, acceptance) and queues the
    # result copy on the runner's copy stream; the host waits for a slot's
    # result only when it reuses the slot, one step later.  The slots are
    # filled once (the synthetic step's inputs do not change), so every
    # replay still moves the full inputs and results across PCIe/C2C.
    step_e2e = None
    if world == 1:
        ropts = {}
        if tree:
            ropts = dict(tree_nodes=cfg.q_len, vocab=W.TREE_ACCEPT_CONFIG["vocab"])
        elif acc is not None:
            ropts = dict(num_draft=cfg.q_len - 1, vocab=W.ACCEPT_CONFIG["vocab"],
                         temperature=acc_opts.get("temperature", 1.0),
                         greedy=acc_opts.get("greedy", False),
                         use_mask="allowed" in acc_opts)
        run = svp.StepRunner(kc, vc, batch=cfg.batch,
                             num_q_heads=cfg.num_q_heads, q_len=cfg.q_len,
                             max_blocks_per_seq=wl.max_blocks_per_seq,
                             n_sink=cfg.n_sink, window=cfg.window, scale=scale,
                             split_pages=args.split_pages,
                             kernel_path=args.kernel_path, **kv_scales, **ropts)
        names = ["q", "k_new", "v_new", "block_table", "seq_lens"]
        src = [q, kn, vn, bt, sl]
        if tree:
            names += ["tree_mask", "target_logits", "draft_logits", "parents",
                      "node_tokens", "uniforms"]
            src += [tm] + list(acc[0])
        elif acc is not None:
            names += ["target_logits", "draft_logits", "draft_tokens", "uniforms"]
            src += list(acc[0])
            if "allowed" in acc_opts:
                names.append("allowed")
                src.append(acc_opts["allowed"])
        for slot in (0, 1):
            for name, t in zip(names, src):
                h = run.host(slot, name)
                a = (t.view(torch.int16).cpu().numpy().view(np.uint16)
                     if t.dtype == torch.bfloat16 else t.cpu().numpy())
                h[...] = a.view(h.dtype) if a.dtype.itemsize == h.dtype.itemsize \
                    and a.dtype.kind != h.dtype.kind else a
        n_run = max(4, min(args.steps, 200))
        for t in range(4):
            if t >= 2:
                run.wait(t % 2)
            run.launch(t % 2)
        run.wait(0)
        run.wait(1)
        r0 = time.perf_counter()
        for t in range(n_run):
            if t >= 2:
                run.wait(t % 2)
            run.launch(t % 2)
        run.wait(0)
        run.wait(1)
        r_ms = (time.perf_counter() - r0) * 1e3 / n_run
        step_bytes_in = sum(run.host(0, n).nbytes for n in names)
        outs = ["out", "lse"] + (["out_tokens", "n_accepted"]
                                 if acc is not None else []) + (
                                     ["out_nodes"] if tree else [])
        step_bytes_out = sum(run.host(0, n).nbytes for n in outs)
        run.close()
        step_e2e = {"value": round(tokens_per_step_of(cfg) / (r_ms / 1e3), 1),
                    "unit": UNIT, "ms_per_step": round(r_ms, 4),
                    "h2d_bytes_per_step": int(step_bytes_in),
                    "d2h_bytes_per_step": int(step_bytes_out)}

    # ---- report ----
    kname, ksrc = attention_kernel(cfg, args.kernel_path)
    tokens_per_step = cfg.batch * cfg.q_len
    value = world * tokens_per_step * args.steps / (ms_max / 1e3)
    attn_avg_s = sum(attn_ms) / len(attn_ms) / 1e3
    peak, peak_kind = measured_peaks()
    achieved = tr["kv_bytes"] / attn_avg_s / 1e9
    plain_e2e = {"value": round(world * tokens_per_step / (e_ms / 1e3), 1),
                 "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                 "d2h_bytes_per_step": int(d2h),
                 "path": "plain public calls, host-synchronised each step"}
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_max / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"f32": "f32", "bf16": "bf16", "fp8": "fp8-e4m3 KV, bf16 q"}[cfg.dtype],
        "data": "synthetic (seeded N(0,1) Q/K/V, shuffled 16-token pages)",
        "config": conf,
        "kv_read_gbs": round(tr["kv_bytes"] * args.steps / (ms / 1e3) / 1e9, 1),
        "attention_us": round(attn_avg_s * 1e6, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} HBM copy bandwidth",
                     "kernel": kname,
                     "traffic": kernel_traffic(kname, ksrc, cfg.name)},
        # end to end: through the graph-captured step (svp_step_*) on one GPU,
        # else the plain calls; both copy each step's inputs from pinned
        # host memory and read its results back
        "e2e": (dict(step_e2e, path="graph-captured step (svp_step)")
                if step_e2e else plain_e2e),
        **({"e2e_plain_calls": plain_e2e} if step_e2e else {}),
        "gpu_launches": int(gpu_launches),
        **({"accept_us": round(sum(acc_ms) / len(acc_ms) * 1e3, 2)}
           if acc is not None else {}),
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# --------------------------------------------------------------------------
# the reference arm: the CPU oracle
# --------------------------------------------------------------------------

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    cfg = W.CONFIGS[args.workload]
    wl = W.make_attention(cfg, poison=False)
    conf, _ = workload_config(wl)
    seqs_per_step = 1
    for i in range(args.warmup):
        oracle_sample(wl, seqs_per_step, start=i)
    t_tot, tok = 0.0, 0
    for i in range(args.steps):
        dt, n = oracle_sample(wl, seqs_per_step, start=args.warmup + i)
        t_tot += dt
        tok += n
    value = tok / t_tot
    sample = (f"each step: {seqs_per_step} of {cfg.batch} sequences of "
              f"{cfg.name}, all heads, fp64 oracle, one thread")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3),
        "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_tot * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": conf,
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": 1,
                         "host_cpus": os.cpu_count(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": UNIT,
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode-7b", choices=sorted(W.CONFIGS))
    ap.add_argument("--split-pages", type=int, default=0,
                    help="pages per split-K unit (0: automatic)")
    ap.add_argument("--kernel-path", type=int, default=0, choices=[0, 1, 2, 3],
                    help="0 automatic, 1 CUDA cores, 2 warp-level tensor "
                         "cores (mma.sync), 3 tcgen05")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's sequence count (smaller "
                         "cases for profiling; reported in config)")
    ap.add_argument("--temperature", type=float, default=1.0,
                    help="verify workloads: sampling temperature of the "
                         "accept step (spec_accept_ex)")
    ap.add_argument("--allowed-density", type=float, default=0.0,
                    help="verify workloads: constrained decoding, each "
                         "token allowed with this probability (0: no mask)")
    ap.add_argument("--greedy", action="store_true",
                    help="verify workloads: greedy (argmax) verification")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time plain API calls instead of CUDA-graph replays")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
