"""Shared test helpers: storage widening and simple layout builders.

Nothing here computes attention or acceptance; the helpers only widen stored
bits to float64 and rearrange pages (labels of physical blocks are arbitrary,
so permuting them together with the table must not change any result).
"""
import numpy as np

from spec_verify_paged_gb300 import workloads as W


def widen(a):
    """Stored values (fp32 or bf16 bits) as float64."""
    if a.dtype == np.uint16:
        return W.bf16_bits_to_f32(a).astype(np.float64)
    return a.astype(np.float64)


def identity_layout(rng, B, Hkv, D, L, dtype="f32", Hq=None, q_len=1):
    """Sequences of equal length L stored contiguously: sequence b owns
    physical blocks b*nblk .. b*nblk+nblk-1 in order, so the logical K of
    (b, g) is simply k_cache[b*nblk:(b+1)*nblk, g].reshape(-1, D)[:L]."""
    Hq = Hq or Hkv
    nblk = -(-L // W.BLOCK_SIZE)
    shape = (B * nblk, Hkv, W.BLOCK_SIZE, D)
    k = W._normals(rng, shape, dtype)
    v = W._normals(rng, shape, dtype)
    q = W._normals(rng, (B, q_len, Hq, D), dtype)
    table = np.arange(B * nblk, dtype=np.int32).reshape(B, nblk)
    seq_lens = np.full((B,), L, np.int32)
    return q, k, v, table, seq_lens


def contiguous_kv(k, v, b, g, L, nblk):
    """Logical rows of (b, g) from an identity layout, float64 [L, D]."""
    D = k.shape[-1]
    kk = widen(k[b * nblk:(b + 1) * nblk, g].reshape(-1, D)[:L])
    vv = widen(v[b * nblk:(b + 1) * nblk, g].reshape(-1, D)[:L])
    return kk, vv


def permute_pages(rng, k, v, table):
    """Relabel physical blocks by a random permutation pi: page i moves to
    slot pi[i] and every table entry follows it."""
    nb = k.shape[0]
    pi = rng.permutation(nb).astype(np.int32)
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[pi] = k
    v2[pi] = v
    t2 = np.where(table >= 0, pi[np.maximum(table, 0)], -1).astype(np.int32)
    return k2, v2, t2


def to_dev(a, device="cuda:0"):
    """numpy -> torch on the GPU; uint16 arrays become bfloat16 (same bits)."""
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_host(t):
    """torch (GPU) -> numpy; bfloat16 comes back as uint16 bit patterns."""
    import torch
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def out_as_f64(t):
    """GPU attention output widened to float64."""
    return widen(to_host(t))


def accept_in_valid_set(out_tokens, n_accepted, draft_tokens, valid):
    """Per sequence: True iff (out_tokens, n_accepted) is one of the outcomes
    in the oracle's valid set (oracle.spec_accept_valid): a reachable path j,
    the first j draft tokens copied, the drawn token among that path's
    candidates, then -1 padding."""
    B, K1 = out_tokens.shape
    ok = np.zeros(B, bool)
    for b in range(B):
        j = int(n_accepted[b])
        if j < 0 or j >= K1 or not valid["path_valid"][b, j]:
            continue
        if not np.array_equal(out_tokens[b, :j], draft_tokens[b, :j]):
            continue
        n = int(valid["n_cand"][b, j])
        if n > valid["cand"].shape[2]:
            continue          # more candidates than listed: undecidable here
        if int(out_tokens[b, j]) not in set(valid["cand"][b, j, :n].tolist()):
            continue
        if np.any(out_tokens[b, j + 1:] != -1):
            continue
        ok[b] = True
    return ok


def tree_accept_in_valid_set(out_tokens, out_nodes, n_accepted, node_tokens,
                             valid):
    """Per sequence: True iff the tree outcome (accepted nodes, their tokens,
    the drawn token, -1 padding) is one of the oracle's valid outcomes
    (oracle.spec_accept_tree_valid)."""
    B, N = out_tokens.shape
    ok = np.zeros(B, bool)
    for b in range(B):
        if valid[b]["n_outcomes"] > len(valid[b]["outcomes"]):
            continue
        k = int(n_accepted[b])
        if k < 0 or k >= N:
            continue
        nodes = tuple(int(x) for x in out_nodes[b, :k])
        if any(n < 0 or n >= N for n in nodes):
            continue
        if not np.array_equal(out_tokens[b, :k], node_tokens[b, list(nodes)]):
            continue
        if np.any(out_nodes[b, k:] != -1) or np.any(out_tokens[b, k + 1:] != -1):
            continue
        tok = int(out_tokens[b, k])
        ok[b] = any(o["nodes"] == nodes and o["n_cand"] == len(o["cand"])
                    and tok in o["cand"] for o in valid[b]["outcomes"])
    return ok


def compare_accept(toks, nacc, ref, valid, draft_tokens, label="spec_accept"):
    """GPU acceptance against the oracle: sequences the oracle does not flag
    must match its outcome exactly; flagged ones (a decision within the band
    of its boundary) must be one of the oracle's valid outcomes.  Returns
    (flagged, flagged and identical to the oracle's own outcome)."""
    near = ref["near_boundary"] != 0
    exact = ((nacc == ref["n_accepted"]) &
             (toks == ref["out_tokens"]).all(axis=1))
    bad_exact = np.nonzero(~near & ~exact)[0]
    inset = accept_in_valid_set(toks, nacc, draft_tokens, valid)
    bad_set = np.nonzero(near & ~inset)[0]
    assert bad_exact.size == 0, (
        f"[{label}] {bad_exact.size} unflagged sequences differ: "
        f"{bad_exact[:8].tolist()}")
    assert bad_set.size == 0, (
        f"[{label}] {bad_set.size} flagged sequences outside the valid set: "
        f"{bad_set[:8].tolist()}")
    # every sequence is in the valid set (the unflagged ones trivially)
    assert inset.all()
    nf = int(near.sum())
    print(f"[{label}] {len(nacc)} sequences: {len(nacc) - nf} identical, "
          f"{nf} flagged near a boundary and inside the valid set "
          f"({int((near & exact).sum())} of them identical)")
    return nf, int((near & exact).sum())


def compare_tree_accept(toks, nodes, nacc, ref, valid, node_tokens,
                        label="spec_accept_tree"):
    """As compare_accept, for tree acceptance."""
    near = ref["near_boundary"] != 0
    exact = ((nacc == ref["n_accepted"]) &
             (toks == ref["out_tokens"]).all(axis=1) &
             (nodes == ref["out_nodes"]).all(axis=1))
    bad_exact = np.nonzero(~near & ~exact)[0]
    inset = tree_accept_in_valid_set(toks, nodes, nacc, node_tokens, valid)
    bad_set = np.nonzero(near & ~inset)[0]
    assert bad_exact.size == 0, (
        f"[{label}] {bad_exact.size} unflagged sequences differ: "
        f"{bad_exact[:8].tolist()}")
    assert bad_set.size == 0, (
        f"[{label}] {bad_set.size} flagged sequences outside the valid set: "
        f"{bad_set[:8].tolist()}")
    assert inset.all()
    nf = int(near.sum())
    print(f"[{label}] {len(nacc)} sequences: {len(nacc) - nf} identical, "
          f"{nf} flagged near a boundary and inside the valid set "
          f"({int((near & exact).sum())} of them identical)")
    return nf, int((near & exact).sum())
