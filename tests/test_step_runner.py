"""The graph-captured decode step (two ping-pong slots, one CUDA graph per
slot, result copies on a separate stream) against the same steps made with
plain calls: outputs, tokens and the final caches must be bit-identical."""
import numpy as np
import pytest

from helpers import to_dev
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


@pytest.mark.parametrize("q_len,num_draft", [(5, 4), (1, 0)])
def test_step_runner_matches_plain_calls(svp, q_len, num_draft):
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
