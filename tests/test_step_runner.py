"""The graph-captured decode step (two ping-pong slots, one CUDA graph per
slot, result copies on a separate stream) against the same steps made with
plain calls: outputs, tokens and the final caches must be bit-identical.
Each step's results, read from the runner's host slots, are also checked
against the fp64 oracle run step by step on its own copy of the caches
(append, attention at the attention tolerances, acceptance exact or inside
the oracle's valid set near a decision boundary)."""
import numpy as np
import pytest

from helpers import compare_accept, compare_tree_accept, to_dev, widen
from spec_verify_paged_gb300 import workloads as W

ATOL, LSE_TOL = 2e-2, 1e-3   # bf16 KV


class _OracleSteps:
    """The oracle's view of a run of steps: its own caches, appended to by
    oracle.kv_append, read by oracle.paged_attention."""

    def __init__(self, oracle_mod, wl):
        self.o = oracle_mod
        self.kc, self.vc = wl.k_cache.copy(), wl.v_cache.copy()
        self.scale = wl.scale

    def attention(self, d, q_len, tree_mask=None):
        self.kc, self.vc = self.o.kv_append(d["k_new"], d["v_new"], self.kc,
                                            self.vc, d["block_table"],
                                            d["seq_lens"])
        if tree_mask is not None:
            return self.o.paged_tree_attention(
                d["q"], self.kc, self.vc, d["block_table"], d["seq_lens"],
                q_len, tree_mask, self.scale)
        return self.o.paged_attention(d["q"], self.kc, self.vc,
                                      d["block_table"], d["seq_lens"], q_len,
                                      0, 0, self.scale)


def _check_attention(got, out_ref, lse_ref):
    err = np.abs(widen(got["out"]) - out_ref).max()
    assert err <= ATOL, err
    if "lse" in got:
        lerr = np.abs(got["lse"].astype(np.float64) - lse_ref).max()
        assert lerr <= LSE_TOL, lerr

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


@pytest.mark.parametrize("q_len,num_draft", [(5, 4), (1, 0)])
def test_step_runner_matches_plain_calls(svp, oracle_mod, q_len, num_draft):
    import torch
    cfg = W.small_config(batch=4, num_q_heads=16, num_kv_heads=4,
                         head_dim=128, q_len=q_len, dtype="bf16", ctx_min=40,
                         ctx_max=300, seed=120 + q_len)
    wl = W.make_attention(cfg, n_new=q_len)
    V = 2000
    steps = 5
    rng = np.random.default_rng(7)
    inputs = []
    for t in range(steps):
        d = {"q": W._normals(rng, wl.q.shape, "bf16"),
             "k_new": W._normals(rng, wl.k_new.shape, "bf16"),
             "v_new": W._normals(rng, wl.v_new.shape, "bf16"),
             "block_table": wl.block_table, "seq_lens": wl.seq_lens}
        if num_draft:
            a = W.make_accept(batch=4, num_draft=num_draft, vocab=V, seed=300 + t)
            d.update(target_logits=a.target_logits, draft_logits=a.draft_logits,
                     draft_tokens=a.draft_tokens, uniforms=a.uniforms)
        inputs.append(d)

    kc1, vc1 = to_dev(wl.k_cache), to_dev(wl.v_cache)
    kc2, vc2 = to_dev(wl.k_cache), to_dev(wl.v_cache)
    run = svp.StepRunner(kc1, vc1, batch=4, num_q_heads=16, q_len=q_len,
                         max_blocks_per_seq=wl.max_blocks_per_seq,
                         scale=float(wl.scale), num_draft=num_draft, vocab=V)
    got = []

    def collect(slot):
        run.wait(slot)
        r = {"out": run.host(slot, "out").copy(), "lse": run.host(slot, "lse").copy()}
        if num_draft:
            r["out_tokens"] = run.host(slot, "out_tokens").copy()
            r["n_accepted"] = run.host(slot, "n_accepted").copy()
        got.append(r)

    for t in range(steps):
        slot = t % 2
        if t >= 2:
            collect(slot)          # step t-2's results, then the slot is free
        for name, arr in inputs[t].items():
            run.host(slot, name)[...] = arr
        run.launch(slot)
    for t in range(max(0, steps - 2), steps):
        collect(t % 2)

    ref = []
    for d in inputs:
        bt, sl = to_dev(d["block_table"]), to_dev(d["seq_lens"])
        svp.kv_append(to_dev(d["k_new"]), to_dev(d["v_new"]), kc2, vc2, bt, sl)
        out, lse = svp.paged_decode_attention(to_dev(d["q"]), kc2, vc2, bt, sl,
                                              q_len=q_len,
                                              scale=float(wl.scale))
        r = {"out": out.view(torch.int16).cpu().numpy().view(np.uint16),
             "lse": lse.cpu().numpy()}
        if num_draft:
            toks, nacc = svp.spec_accept(to_dev(d["target_logits"]),
                                         to_dev(d["draft_logits"]),
                                         to_dev(d["draft_tokens"]),
                                         to_dev(d["uniforms"]))
            r["out_tokens"] = toks.cpu().numpy()
            r["n_accepted"] = nacc.cpu().numpy()
        ref.append(r)
    torch.cuda.synchronize()
    assert len(got) == steps
    for t in range(steps):
        for k in ref[t]:
            assert np.array_equal(got[t][k], ref[t][k]), (t, k)
    # bitwise: unused cache rows hold NaN poison, which == would reject
    assert torch.equal(kc1.view(torch.int16), kc2.view(torch.int16))
    assert torch.equal(vc1.view(torch.int16), vc2.view(torch.int16))
    run.close()
    assert svp.read_device_status() == 0
    # the runner's host-slot results against the oracle, step by step
    ora = _OracleSteps(oracle_mod, wl)
    for t, d in enumerate(inputs):
        out_ref, lse_ref = ora.attention(d, q_len)
        _check_attention(got[t], out_ref, lse_ref)
        if num_draft:
            ref = oracle_mod.spec_accept(d["target_logits"], d["draft_logits"],
                                         d["draft_tokens"], d["uniforms"])
            valid = oracle_mod.spec_accept_valid(
                d["target_logits"], d["draft_logits"], d["draft_tokens"],
                d["uniforms"])
            compare_accept(got[t]["out_tokens"], got[t]["n_accepted"], ref,
                           valid, d["draft_tokens"], label=f"runner step {t}")
    # and the runner's cache after the last step holds the oracle's appends
    assert np.array_equal(kc1.view(torch.int16).cpu().numpy().view(np.uint16),
                          ora.kc)


def _run_steps(run, inputs, fields_out):
    """Feeds `inputs` through the two slots (one step ahead) and returns each
    step's outputs."""
    got = []

    def collect(slot):
        run.wait(slot)
        got.append({k: run.host(slot, k).copy() for k in fields_out})

    steps = len(inputs)
    for t in range(steps):
        slot = t % 2
        if t >= 2:
            collect(slot)
        for name, arr in inputs[t].items():
            run.host(slot, name)[...] = arr
        run.launch(slot)
    for t in range(max(0, steps - 2), steps):
        collect(t % 2)
    return got


def test_step_runner_tree_matches_plain_calls(svp, oracle_mod):
    """A draft-tree step (tree attention + tree acceptance) through the
    runner equals the same steps made with plain calls."""
    import torch
    N = 7
    par = W.binary_tree_parents(2)
    cfg = W.small_config(batch=3, num_q_heads=16, num_kv_heads=4,
                         head_dim=128, q_len=N, dtype="bf16", ctx_min=N + 30,
                         ctx_max=400, seed=131)
    wl = W.make_attention(cfg, n_new=N)
    V = 1500
    rng = np.random.default_rng(8)
    inputs = []
    for t in range(4):
        a = W.make_tree_accept(batch=3, vocab=V, seed=400 + t, parents=par)
        inputs.append({
            "q": W._normals(rng, wl.q.shape, "bf16"),
            "k_new": W._normals(rng, wl.k_new.shape, "bf16"),
            "v_new": W._normals(rng, wl.v_new.shape, "bf16"),
            "block_table": wl.block_table, "seq_lens": wl.seq_lens,
            "tree_mask": W.tree_mask_from_parents(a.parents),
            "target_logits": a.target_logits, "draft_logits": a.draft_logits,
            "parents": a.parents, "node_tokens": a.node_tokens,
            "uniforms": a.uniforms})
    kc1, vc1 = to_dev(wl.k_cache), to_dev(wl.v_cache)
    kc2, vc2 = to_dev(wl.k_cache), to_dev(wl.v_cache)
    run = svp.StepRunner(kc1, vc1, batch=3, num_q_heads=16, q_len=N,
                         max_blocks_per_seq=wl.max_blocks_per_seq,
                         scale=float(wl.scale), vocab=V, tree_nodes=N)
    outs = ("out", "lse", "out_tokens", "out_nodes", "n_accepted")
    got = _run_steps(run, inputs, outs)
    for t, d in enumerate(inputs):
        bt, sl = to_dev(d["block_table"]), to_dev(d["seq_lens"])
        svp.kv_append(to_dev(d["k_new"]), to_dev(d["v_new"]), kc2, vc2, bt, sl)
        out, lse = svp.paged_tree_attention(
            to_dev(d["q"]), kc2, vc2, bt, sl,
            to_dev(d["tree_mask"].view(np.int32)), scale=float(wl.scale))
        toks, nodes, nacc = svp.spec_accept_tree(
            to_dev(d["target_logits"]), to_dev(d["draft_logits"]),
            to_dev(d["parents"]), to_dev(d["node_tokens"]),
            to_dev(d["uniforms"]))
        ref = {"out": out.view(torch.int16).cpu().numpy().view(np.uint16),
               "lse": lse.cpu().numpy(), "out_tokens": toks.cpu().numpy(),
               "out_nodes": nodes.cpu().numpy(), "n_accepted": nacc.cpu().numpy()}
        for k in outs:
            assert np.array_equal(got[t][k], ref[k]), (t, k)
    torch.cuda.synchronize()
    assert torch.equal(kc1.view(torch.int16), kc2.view(torch.int16))
    run.close()
    assert svp.read_device_status() == 0
    ora = _OracleSteps(oracle_mod, wl)
    for t, d in enumerate(inputs):
        out_ref, lse_ref = ora.attention(d, N, tree_mask=d["tree_mask"])
        _check_attention(got[t], out_ref, lse_ref)
        ref = oracle_mod.spec_accept_tree(d["target_logits"], d["draft_logits"],
                                          d["parents"], d["node_tokens"],
                                          d["uniforms"])
        valid = oracle_mod.spec_accept_tree_valid(
            d["target_logits"], d["draft_logits"], d["parents"],
            d["node_tokens"], d["uniforms"])
        compare_tree_accept(got[t]["out_tokens"], got[t]["out_nodes"],
                            got[t]["n_accepted"], ref, valid, d["node_tokens"],
                            label=f"runner tree step {t}")


@pytest.mark.parametrize("opts", [dict(temperature=0.7, use_mask=True),
                                  dict(greedy=True), dict(temperature=1.6)])
def test_step_runner_epilogue_matches_plain_calls(svp, oracle_mod, opts):
    """The verify epilogue (temperature, token mask, greedy) through the
    runner equals spec_accept with the same options."""
    import torch
    K, V = 4, 3000
    cfg = W.small_config(batch=4, num_q_heads=16, num_kv_heads=4,
                         head_dim=128, q_len=K + 1, dtype="bf16", ctx_min=40,
                         ctx_max=300, seed=141)
    wl = W.make_attention(cfg, n_new=K + 1)
    rng = np.random.default_rng(9)
    words = (V + 31) // 32
    inputs = []
    for t in range(4):
        a = W.make_accept(batch=4, num_draft=K, vocab=V, seed=500 + t)
        d = {"q": W._normals(rng, wl.q.shape, "bf16"),
             "k_new": W._normals(rng, wl.k_new.shape, "bf16"),
             "v_new": W._normals(rng, wl.v_new.shape, "bf16"),
             "block_table": wl.block_table, "seq_lens": wl.seq_lens,
             "target_logits": a.target_logits, "draft_logits": a.draft_logits,
             "draft_tokens": a.draft_tokens, "uniforms": a.uniforms}
        if opts.get("use_mask"):
            d["allowed"] = rng.integers(0, 2**32, size=(4, K + 1, words),
                                        dtype=np.uint64).astype(np.uint32)
            d["allowed"][..., 0] |= 1   # token 0 always allowed
        inputs.append(d)
    kc1, vc1 = to_dev(wl.k_cache), to_dev(wl.v_cache)
    kc2, vc2 = to_dev(wl.k_cache), to_dev(wl.v_cache)
    run = svp.StepRunner(kc1, vc1, batch=4, num_q_heads=16, q_len=K + 1,
                         max_blocks_per_seq=wl.max_blocks_per_seq,
                         scale=float(wl.scale), num_draft=K, vocab=V, **opts)
    outs = ("out", "out_tokens", "n_accepted")
    got = _run_steps(run, inputs, outs)
    for t, d in enumerate(inputs):
        bt, sl = to_dev(d["block_table"]), to_dev(d["seq_lens"])
        svp.kv_append(to_dev(d["k_new"]), to_dev(d["v_new"]), kc2, vc2, bt, sl)
        out, _ = svp.paged_decode_attention(to_dev(d["q"]), kc2, vc2, bt, sl,
                                            q_len=K + 1, scale=float(wl.scale))
        allowed = (to_dev(d["allowed"].view(np.int32))
                   if "allowed" in d else None)
        toks, nacc = svp.spec_accept(
            to_dev(d["target_logits"]), to_dev(d["draft_logits"]),
            to_dev(d["draft_tokens"]), to_dev(d["uniforms"]),
            temperature=opts.get("temperature", 1.0), allowed=allowed,
            greedy=opts.get("greedy", False))
        ref = {"out": out.view(torch.int16).cpu().numpy().view(np.uint16),
               "out_tokens": toks.cpu().numpy(), "n_accepted": nacc.cpu().numpy()}
        for k in outs:
            assert np.array_equal(got[t][k], ref[k]), (t, k)
    run.close()
    assert svp.read_device_status() == 0
    ora = _OracleSteps(oracle_mod, wl)
    T = opts.get("temperature", 1.0)
    greedy = opts.get("greedy", False)
    for t, d in enumerate(inputs):
        out_ref, lse_ref = ora.attention(d, K + 1)
        _check_attention(got[t], out_ref, lse_ref)
        allowed = d.get("allowed")
        ref = oracle_mod.spec_accept_ex(d["target_logits"], d["draft_logits"],
                                        d["draft_tokens"], d["uniforms"],
                                        temperature=T, allowed=allowed,
                                        greedy=greedy)
        if greedy:
            assert np.array_equal(got[t]["out_tokens"], ref["out_tokens"])
            assert np.array_equal(got[t]["n_accepted"], ref["n_accepted"])
            continue
        valid = oracle_mod.spec_accept_valid(
            d["target_logits"], d["draft_logits"], d["draft_tokens"],
            d["uniforms"], temperature=T, allowed=allowed)
        compare_accept(got[t]["out_tokens"], got[t]["n_accepted"], ref, valid,
                       d["draft_tokens"], label=f"runner epilogue step {t}")
