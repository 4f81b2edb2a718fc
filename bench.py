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
NOMINAL_HBM_GBS = 8000.0   # the ~8 TB/s HBM roofline of a GB300
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

def accept_inputs(cfg):
    """The acceptance step's inputs of a verify workload (K = q_len - 1
    drafts, vocab 32,000, same seed as the attention inputs), a draft tree's
    for the tree workload, None for plain decode."""
    if cfg.tree_depth > 0:
        return W.make_tree_accept(batch=cfg.batch, depth=cfg.tree_depth,
                                  vocab=W.TREE_ACCEPT_CONFIG["vocab"],
                                  seed=cfg.seed)
    if cfg.q_len > 1:
        return W.make_accept(batch=cfg.batch, num_draft=cfg.q_len - 1,
                             vocab=W.ACCEPT_CONFIG["vocab"], seed=cfg.seed)
    return None


def oracle_sample(wl, n_seqs, start=0, awl=None):
    """Run the fp64 oracle on n_seqs sequences of the workload (all heads,
    all query rows, and the acceptance of those sequences when awl is
    given); returns (seconds, query tokens)."""
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
    if awl is not None:
        s = np.array(seqs)
        if wl.cfg.tree_depth > 0:
            oracle.spec_accept_tree(awl.target_logits[s], awl.draft_logits[s],
                                    awl.parents[s], awl.node_tokens[s],
                                    awl.uniforms[s])
        else:
            oracle.spec_accept(awl.target_logits[s], awl.draft_logits[s],
                               awl.draft_tokens[s], awl.uniforms[s])
    return time.perf_counter() - t, n_seqs * wl.q_len


def cpu_baseline(wl, awl=None, budget_s=10.0, max_passes=20):
    """The oracle as it stands, single-threaded, on whole sequences of the
    workload (cycling through them) until about budget_s seconds of CPU
    work (at least one sequence)."""
    total_t, total_tok, n = 0.0, 0, 0
    while (n == 0 or total_t < budget_s) and n < max_passes * wl.cfg.batch:
        dt, tok = oracle_sample(wl, 1, start=n, awl=awl)
        total_t += dt
        total_tok += tok
        n += 1
    what = "attention" + (" and acceptance" if awl is not None else "")
    return {"value": total_tok / total_t, "unit": UNIT, "cores": 1,
            "host_cpus": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{n} sequence passes over the {wl.cfg.batch} sequences "
                      f"of {wl.cfg.name} ({what}, all {wl.cfg.num_q_heads} "
                      f"heads, fp64, one thread), {total_t:.1f} s"}


def accept_boundary(cfg, awl, toks, nodes, nacc):
    """The fp64 oracle's view of the acceptance step the GPU just made (part
    of the CPU-baseline leg): how many sequences have a decision within 1e-6
    of its boundary, and whether every GPU outcome is the oracle's or, for
    a flagged sequence, one of the outcomes the oracle lists as valid."""
    import oracle
    oracle.build()
    t = time.perf_counter()
    if cfg.tree_depth > 0:
        ref = oracle.spec_accept_tree(awl.target_logits, awl.draft_logits,
                                      awl.parents, awl.node_tokens,
                                      awl.uniforms)
        valid = oracle.spec_accept_tree_valid(
            awl.target_logits, awl.draft_logits, awl.parents,
            awl.node_tokens, awl.uniforms)
        same = ((nacc == ref["n_accepted"]) &
                (toks == ref["out_tokens"]).all(1) &
                (nodes == ref["out_nodes"]).all(1))
        inset = []
        for b in range(cfg.batch):
            k = int(nacc[b])
            path = tuple(int(x) for x in nodes[b, :max(k, 0)])
            inset.append(any(o["nodes"] == path and int(toks[b, k]) in o["cand"]
                             for o in valid[b]["outcomes"]) if k >= 0 else False)
    else:
        ref = oracle.spec_accept(awl.target_logits, awl.draft_logits,
                                 awl.draft_tokens, awl.uniforms)
        valid = oracle.spec_accept_valid(awl.target_logits, awl.draft_logits,
                                         awl.draft_tokens, awl.uniforms)
        same = ((nacc == ref["n_accepted"]) &
                (toks == ref["out_tokens"]).all(1))
        inset = []
        for b in range(cfg.batch):
            j = int(nacc[b])
            ok = 0 <= j < toks.shape[1] and bool(valid["path_valid"][b, j])
            ok = ok and np.array_equal(toks[b, :j], awl.draft_tokens[b, :j])
            ok = ok and int(toks[b, j]) in valid["cand"][b, j].tolist()
            inset.append(ok)
    near = ref["near_boundary"] != 0
    return {"sequences": int(cfg.batch), "boundary_draws": int(near.sum()),
            "identical_to_oracle": int(same.sum()),
            "flagged_inside_valid_set": int((near & np.array(inset)).sum()),
            "unflagged_mismatches": int((~near & ~same).sum()),
            "oracle_n_accepted_hist": np.bincount(
                ref["n_accepted"], minlength=toks.shape[1]).tolist(),
            "oracle_s": round(time.perf_counter() - t, 3)}


def tokens_per_step_of(cfg):
    return cfg.batch * cfg.q_len


def workload_config(wl, args=None):
    """The `config` object of a bench line; both arms emit the same one."""
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
         "l2": ("no flush: each step reads %.2f GB of KV, > 129 MB L2"
                % (tr["kv_bytes"] / 1e9)) if tr["kv_bytes"] > 129e6 else
               ("no flush: the %.1f MB of KV stay L2-resident (a latency-bound "
                "case)" % (tr["kv_bytes"] / 1e6))}
    if cfg.tree_depth > 0:
        c["draft_tree"] = {"shape": "complete binary", "depth": cfg.tree_depth,
                           "nodes": cfg.q_len}
        c["accept"] = {"batch": cfg.batch, "tree_nodes": cfg.q_len,
                       "vocab": W.TREE_ACCEPT_CONFIG["vocab"]}
    elif cfg.q_len > 1:
        c["accept"] = {"batch": cfg.batch, "num_draft": cfg.q_len - 1,
                       "vocab": W.ACCEPT_CONFIG["vocab"]}
        if args is not None and (args.temperature != 1.0 or args.greedy or
                                 args.allowed_density > 0):
            c["accept"]["epilogue"] = {
                "temperature": args.temperature, "greedy": bool(args.greedy),
                "allowed_density": args.allowed_density}
    if args is not None and args.split_pages:
        c["split_pages"] = args.split_pages
    if args is not None and args.kernel_path:
        c["kernel_path"] = {1: "cuda_cores", 2: "tensor_cores",
                            3: "tcgen05"}[args.kernel_path]
    return c, tr


# --------------------------------------------------------------------------
# the GPU arm
# --------------------------------------------------------------------------

class GpuCase:
    """One workload resident on the device: its step as plain library calls
    and as CUDA graphs (the whole step, and each phase on its own)."""

    def __init__(self, svp, cfg, args, dev):
        import torch
        self.svp, self.cfg, self.args, self.dev = svp, cfg, args, dev
        wl = W.make_attention(cfg, n_new=cfg.q_len, poison=False)
        self.wl = wl
        self.conf, self.tr = workload_config(wl, args)
        self.q = to_dev(wl.q, dev)
        self.kc, self.vc = to_dev(wl.k_cache, dev), to_dev(wl.v_cache, dev)
        self.bt, self.sl = to_dev(wl.block_table, dev), to_dev(wl.seq_lens, dev)
        self.kn, self.vn = to_dev(wl.k_new, dev), to_dev(wl.v_new, dev)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty((cfg.batch, cfg.q_len, cfg.num_q_heads),
                               dtype=torch.float32, device=dev)
        self.tree = cfg.tree_depth > 0
        self.tm = (to_dev(wl.tree_mask.view(np.int32), dev) if self.tree
                   else None)
        self.awl = accept_inputs(cfg)
        self.acc = None
        self.acc_opts = {}
        if self.tree:
            a = self.awl
            acc_in = [to_dev(x, dev) for x in (a.target_logits, a.draft_logits,
                                               a.parents, a.node_tokens,
                                               a.uniforms)]
            acc_out = tuple(torch.empty(shape, dtype=torch.int32, device=dev)
                            for shape in ((cfg.batch, cfg.q_len),
                                          (cfg.batch, cfg.q_len), (cfg.batch,)))
            self.acc = (acc_in, acc_out)
        elif self.awl is not None:
            a = self.awl
            acc_in = [to_dev(x, dev) for x in (a.target_logits, a.draft_logits,
                                               a.draft_tokens, a.uniforms)]
            acc_out = (torch.empty((cfg.batch, cfg.q_len), dtype=torch.int32,
                                   device=dev),
                       torch.empty((cfg.batch,), dtype=torch.int32, device=dev))
            self.acc = (acc_in, acc_out)
            # the verify epilogue: temperature, token mask, greedy
            if args.temperature != 1.0:
                self.acc_opts["temperature"] = args.temperature
            if args.greedy:
                self.acc_opts["greedy"] = True
            if args.allowed_density > 0:
                V = W.ACCEPT_CONFIG["vocab"]
                mrng = np.random.default_rng(cfg.seed + 7)
                allowed = mrng.random((cfg.batch, cfg.q_len, V)) < args.allowed_density
                allowed[..., 0] = True
                words = (V + 31) // 32
                pad = np.zeros((cfg.batch, cfg.q_len, words * 32), bool)
                pad[..., :V] = allowed
                bits = np.packbits(pad, axis=-1, bitorder="little").view(np.int32)
                self.acc_opts["allowed"] = to_dev(np.ascontiguousarray(bits), dev)
        self.stream = torch.cuda.current_stream(dev)
        self.scale = float(wl.scale)
        # an FP8 cache's scales (1 otherwise)
        self.kv_scales = dict(k_scale=wl.k_scale, v_scale=wl.v_scale)
        self.launches = 0
        self.graphs = None

    # -- the library calls of one step --
    def attn_call(self, q_, bt_, sl_, out_, lse_, tm_=None):
        a, cfg = self.args, self.cfg
        if self.tree:
            self.svp.paged_tree_attention(
                q_, self.kc, self.vc, bt_, sl_, tm_, scale=self.scale,
                out=out_, lse=lse_, split_pages=a.split_pages,
                kernel_path=a.kernel_path, **self.kv_scales)
        else:
            self.svp.paged_decode_attention(
                q_, self.kc, self.vc, bt_, sl_, q_len=cfg.q_len,
                n_sink=cfg.n_sink, window=cfg.window, scale=self.scale,
                out=out_, lse=lse_, split_pages=a.split_pages,
                kernel_path=a.kernel_path, **self.kv_scales)

    def accept_with(self, inputs, outputs, opts=None):
        opts = self.acc_opts if opts is None else opts
        if self.tree:
            self.svp.spec_accept_tree(*inputs, out_tokens=outputs[0],
                                      out_nodes=outputs[1],
                                      n_accepted=outputs[2])
        else:
            self.svp.spec_accept(*inputs, out_tokens=outputs[0],
                                 n_accepted=outputs[1], **opts)

    def append_call(self):
        self.svp.kv_append(self.kn, self.vn, self.kc, self.vc, self.bt,
                           self.sl, **self.kv_scales)

    def plain_step(self, ev=None):
        svp = self.svp
        self.append_call()
        n = svp.last_launch_count()
        if ev is not None:
            ev[0].record(self.stream)
        self.attn_call(self.q, self.bt, self.sl, self.out, self.lse, self.tm)
        n += svp.last_launch_count()
        if ev is not None:
            ev[1].record(self.stream)
        if self.acc is not None:
            self.accept_with(self.acc[0], self.acc[1])
            n += svp.last_launch_count()
            if ev is not None:
                ev[2].record(self.stream)
        self.launches += n

    # -- CUDA graphs: the whole step, and the step cut short --
    def capture(self):
        """The library keeps no per-call state, so a replay does exactly the
        work of a call.  Inside one graph each kernel is a programmatic
        dependent launch of the one before.  Besides the whole step, two
        prefixes of it are captured -- the append alone, and the append
        with the attention call -- so that each phase's cost is measured as
        what it adds to the step, with the same launches and overlaps as in
        the step itself."""
        import torch
        svp = self.svp
        g_step, g_app, g_noacc = (torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(),
                                  torch.cuda.CUDAGraph())
        with torch.cuda.graph(g_app):
            self.append_call()
        n_app = svp.last_launch_count()
        with torch.cuda.graph(g_noacc):
            self.append_call()
            self.attn_call(self.q, self.bt, self.sl, self.out, self.lse,
                           self.tm)
        n_attn = svp.last_launch_count()
        n_acc = 0
        with torch.cuda.graph(g_step):
            self.append_call()
            self.attn_call(self.q, self.bt, self.sl, self.out, self.lse,
                           self.tm)
            if self.acc is not None:
                self.accept_with(self.acc[0], self.acc[1])
                n_acc = svp.last_launch_count()
        torch.cuda.synchronize(self.dev)
        self.graphs = (g_step, g_app, g_noacc if self.acc is not None else None)
        self.n_launch = (n_app, n_attn, n_acc)

    def whole_step(self):
        self.graphs[0].replay()
        self.launches += sum(self.n_launch)

    def warm_graphs(self):
        g_step, g_app, g_noacc = self.graphs
        for g in (g_step, g_app, g_noacc):
            if g is not None:
                g.replay()

    def measure(self, steps, sampler, world=1, use_graph=True):
        """Times `steps` steps (graph replays of the whole step, or plain
        calls).  With graphs, two more timed loops replay the step's
        prefixes (append alone; append and attention), `steps` times each:
        attention = t(append + attention) - t(append), acceptance =
        t(step) - t(append + attention), per step."""
        import torch
        import torch.distributed as dist
        ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3))
              for _ in range(steps)]
        ep = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        self.launches = 0
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(self.dev)
        t0 = time.time()
        start.record(self.stream)
        for i in range(steps):
            if use_graph:
                self.whole_step()
            else:
                self.plain_step(ev[i])
        end.record(self.stream)
        if use_graph:  # the step's prefixes, in two more timed loops
            _, g_app, g_noacc = self.graphs
            n_app, n_attn, _ = self.n_launch
            ep[0].record(self.stream)
            for _ in range(steps):
                g_app.replay()
            ep[1].record(self.stream)
            if g_noacc is not None:
                for _ in range(steps):
                    g_noacc.replay()
            ep[2].record(self.stream)
            self.launches += steps * (n_app + (n_app + n_attn
                                               if g_noacc is not None else 0))
        torch.cuda.synchronize(self.dev)
        t1 = time.time()
        if world > 1:
            dist.barrier()
        ms = start.elapsed_time(end)
        if use_graph:
            t_app = ep[0].elapsed_time(ep[1]) / steps
            t_step = ms / steps
            if self.acc is not None:
                t_noacc = ep[1].elapsed_time(ep[2]) / steps
                attn_ms = [t_noacc - t_app]
                acc_ms = [t_step - t_noacc]
            else:
                attn_ms = [t_step - t_app]
                acc_ms = None
        else:
            attn_ms = [e[0].elapsed_time(e[1]) for e in ev]
            acc_ms = ([e[1].elapsed_time(e[2]) for e in ev]
                      if self.acc is not None else None)
        return {"ms": ms, "attn_ms": attn_ms, "acc_ms": acc_ms,
                "launches": self.launches, "t0": t0, "t1": t1}

    def accept_results(self):
        """(tokens, nodes or None, n_accepted) of the last acceptance call."""
        if self.acc is None:
            return None
        outs = [t.cpu().numpy() for t in self.acc[1]]
        if self.tree:
            return outs[0], outs[1], outs[2]
        return outs[0], None, outs[1]

    def free(self):
        import torch
        for k in list(self.__dict__):
            if k not in ("cfg", "conf", "tr", "args"):
                setattr(self, k, None)
        torch.cuda.empty_cache()


def roofline_of(case, attn_avg_s):
    cfg = case.cfg
    kname, ksrc = attention_kernel(cfg, case.args.kernel_path)
    peak, peak_kind = measured_peaks()
    achieved = case.tr["kv_bytes"] / attn_avg_s / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1),
            "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "frac_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
            "peak_source": f"{peak_kind} HBM copy bandwidth (frac); "
                           f"frac_8tbs against the nominal 8 TB/s",
            "kernel": kname,
            "traffic": kernel_traffic(kname, ksrc, cfg.name)}


def accept_summary(case):
    """The acceptance step's own output: the n_accepted histogram of the
    batch (path length for a draft tree)."""
    r = case.accept_results()
    if r is None:
        return None
    toks, nodes, nacc = r
    return {"n_accepted_hist": np.bincount(np.maximum(nacc, 0),
                                           minlength=case.cfg.q_len).tolist(),
            "mean_accepted": round(float(nacc.mean()), 3),
            "tokens_per_sequence": round(float(nacc.mean()) + 1.0, 3)}


def measure_other_workload(svp, name, args, dev):
    """One entry of the `workloads` object: the workload's step replayed as
    one CUDA graph long enough for the clock sampler (>= 0.3 s, >= 50
    steps), its phase times, roofline fractions, clocks, acceptance
    histogram and, on the CPU-baseline leg, the oracle's rate and its view
    of the acceptance step."""
    import torch
    cfg = W.CONFIGS[name]
    case = GpuCase(svp, cfg, args, dev)
    for _ in range(args.warmup):
        case.plain_step()
    torch.cuda.synchronize(dev)
    assert svp.read_device_status() == 0, f"{name}: device status flags raised"
    case.capture()
    for _ in range(3):
        case.warm_graphs()
    # size the timed loop from a short probe
    probe = case.measure(10, None)
    per_step_s = max(probe["ms"] / 10 / 1e3, 1e-6)
    steps = int(min(20000, max(50, math.ceil(0.3 / per_step_s))))
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    time.sleep(0.3)
    m = case.measure(steps, sampler)
    time.sleep(0.1)
    sampler.stop()
    attn_avg_s = sum(m["attn_ms"]) / len(m["attn_ms"]) / 1e3
    roof = roofline_of(case, attn_avg_s)
    e = {"config": case.conf, "steps": steps,
         "ms_per_step": round(m["ms"] / steps, 5),
         "value": round(tokens_per_step_of(cfg) * steps / (m["ms"] / 1e3), 1),
         "unit": UNIT,
         "attention_us": round(attn_avg_s * 1e6, 2),
         "kv_bytes": int(case.tr["kv_bytes"]),
         "kv_read_gbs": roof["achieved"],
         "frac": roof["frac"], "frac_8tbs": roof["frac_8tbs"],
         "kernel": roof["kernel"], "traffic": roof["traffic"],
         "gpu_launches": int(m["launches"]),
         "clocks": sampler.summary(m["t0"], m["t1"])}
    if m["acc_ms"] is not None:
        e["accept_us"] = round(sum(m["acc_ms"]) / len(m["acc_ms"]) * 1e3, 2)
        e["accept"] = accept_summary(case)
    if not args.no_cpu_baseline:
        e["cpu_baseline"] = cpu_baseline(case.wl, case.awl, budget_s=2.0)
        if case.acc is not None:
            toks, nodes, nacc = case.accept_results()
            e["cpu_baseline"]["accept_check"] = accept_boundary(
                cfg, case.awl, toks, nodes, nacc)
    case.free()
    return e


OTHER_WORKLOADS = ("long-context-128k", "long-context-128k-verify",
                   "verify-gqa", "stream-sink-window", "tiny-decode",
                   "decode-7b-fp8", "tree-verify")


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
    case = GpuCase(svp, cfg, args, dev)
    conf, tr = case.conf, case.tr
    if args.batch:
        conf["batch_override"] = args.batch
    timing = ("plain calls" if args.no_graph else
              "one CUDA graph per step (append, attention, acceptance as "
              "programmatic dependent launches); phase times are what each "
              "phase adds to the step: two more timed loops replay the "
              "step's prefixes (append; append + attention)")

    for _ in range(args.warmup):
        case.plain_step()
    torch.cuda.synchronize(dev)
    assert svp.read_device_status() == 0, "device status flags raised"

    # The timed loop replays the step as one CUDA graph captured once here:
    # a step of tens of microseconds would otherwise be paced by the host's
    # Python and launch overhead, not by the GPU.  The phase times
    # (attention call, acceptance call) come from a second timed loop that
    # replays each phase as its own graph with CUDA events between them.
    if not args.no_graph:
        case.capture()
        for _ in range(3):
            case.warm_graphs()
        torch.cuda.synchronize(dev)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)  # let the sampler start producing lines
    m = case.measure(args.steps, sampler, world, use_graph=not args.no_graph)
    time.sleep(0.1)
    sampler.stop()
    clocks = sampler.summary(m["t0"], m["t1"])
    ms = m["ms"]
    ms_max = max_over_ranks(ms, world)
    gpu_launches = m["launches"]
    q, kc, vc, bt, sl = case.q, case.kc, case.vc, case.bt, case.sl
    kn, vn, tm, acc, acc_opts = case.kn, case.vn, case.tm, case.acc, case.acc_opts
    tree, stream, scale = case.tree, case.stream, case.scale
    out, lse, kv_scales = case.out, case.lse, case.kv_scales
    acc_stats = accept_summary(case)

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
        case.attn_call(d_views["q"], d_views["block_table"],
                       d_views["seq_lens"], r_views["out"], r_views["lse"],
                       d_views.get("tree_mask"))
        if acc is not None:
            e2e_opts = dict(acc_opts)
            if "allowed" in e2e_opts:
                e2e_opts["allowed"] = d_views["allowed"]
            case.accept_with([d_views[k] for k in acc_names],
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
    # replay still moves the full inputs and results across the host link.
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
                             max_blocks_per_seq=case.wl.max_blocks_per_seq,
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
    tokens_per_step = cfg.batch * cfg.q_len
    value = world * tokens_per_step * args.steps / (ms_max / 1e3)
    attn_avg_s = sum(m["attn_ms"]) / len(m["attn_ms"]) / 1e3
    roof = roofline_of(case, attn_avg_s)
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
        "timing": timing,
        "kv_read_gbs": round(tr["kv_bytes"] * args.steps / (ms / 1e3) / 1e9, 1),
        "attention_us": round(attn_avg_s * 1e6, 2),
        "roofline": roof,
        # end to end: through the graph-captured step (svp_step_*) on one GPU,
        # else the plain calls; both copy each step's inputs from pinned
        # host memory and read its results back
        "e2e": (dict(step_e2e, path="graph-captured step (svp_step)")
                if step_e2e else plain_e2e),
        **({"e2e_plain_calls": plain_e2e} if step_e2e else {}),
        "gpu_launches": int(gpu_launches),
        **({"accept_us": round(sum(m["acc_ms"]) / len(m["acc_ms"]) * 1e3, 2),
            "accept": acc_stats}
           if acc is not None else {}),
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case.wl, case.awl)
        if acc is not None:
            toks, nodes, nacc = case.accept_results()
            line["cpu_baseline"]["accept_check"] = accept_boundary(
                cfg, case.awl, toks, nodes, nacc)
    case.free()
    del q, kc, vc, bt, sl, kn, vn, tm, acc, acc_opts, out, lse
    del h_in, d_in, d_views, h_res, d_res, r_views
    torch.cuda.empty_cache()
    # every other workload at one GPU, same build, same process
    if world == 1 and not args.no_workloads and not args.batch:
        others = {}
        for name in OTHER_WORKLOADS:
            if name == cfg.name:
                continue
            others[name] = measure_other_workload(svp, name, args, dev)
        line["workloads"] = others
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
    awl = accept_inputs(cfg)
    conf, _ = workload_config(wl, args)
    seqs_per_step = 1
    for i in range(args.warmup):
        oracle_sample(wl, seqs_per_step, start=i, awl=awl)
    t_tot, tok = 0.0, 0
    for i in range(args.steps):
        dt, n = oracle_sample(wl, seqs_per_step, start=args.warmup + i, awl=awl)
        t_tot += dt
        tok += n
    value = tok / t_tot
    sample = (f"each step: {seqs_per_step} of {cfg.batch} sequences of "
              f"{cfg.name}, all heads" +
              (", with its acceptance" if awl is not None else "") +
              ", fp64 oracle, one thread")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3),
        "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_tot * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": conf,
        "timing": "host wall clock around each oracle call",
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
    ap.add_argument("--no-workloads", action="store_true",
                    help="measure the named workload only (no `workloads` "
                         "object with the other configurations)")
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
