"""A model of the CUDA-core attention kernel's page ring, run under random
interleavings on the CPU.

The producer warp copies the pages of a segment, in order, into a ring of
STAGES shared-memory stages (page c into stage c mod STAGES, after the
stage's previous page was released); NSTREAM consumer streams take the
pages round-robin (stream k: pages k, k + NSTREAM, ...), each waiting with a
parity test on the stage's "full" barrier and releasing the stage when it
holds the page in registers.  A parity wait cannot tell phase n from phase
n + 2.  When STAGES is a multiple of NSTREAM, the previous page of a stage
belongs to the same stream, which has waited for it already, so no wait is
ever two phases ahead; otherwise a stream can pass its wait two phases
early and consume a stage whose copy has not landed.  The kernel refuses to
compile unless STAGES % NSTREAM == 0; this model shows why.
"""
import random

import pytest


class Bar:
    def __init__(self):
        self.done = 0          # completed phases

    def test(self, parity):
        return (self.done & 1) != parity


def run(seed, stages, nstream, pages=40):
    """Returns None if every stream read the page it waited for and the
    run completed, else a description of the first early pass (or of a
    run that stopped making progress: an early release can also leave the
    producer waiting on a phase that has already gone by)."""
    rnd = random.Random(seed)
    full = [Bar() for _ in range(stages)]
    empty = [Bar() for _ in range(stages)]
    holds = [None] * stages        # page whose copy has landed in a stage
    inflight = []                  # (stage, page) copies issued, not landed
    produced = 0
    nxt = list(range(nstream))     # next page of each stream
    for _ in range(40_000):
        if all(n >= pages for n in nxt):
            return None
        actor = rnd.randrange(nstream + 2)
        if actor == nstream:       # producer: issue the next page's copy
            c = produced
            if c < pages:
                s = c % stages
                if c < stages or empty[s].test(((c // stages) & 1) ^ 1):
                    inflight.append((s, c))
                    produced += 1
        elif actor == nstream + 1:  # a copy lands (often the newest first)
            if inflight:
                i = len(inflight) - 1 if rnd.random() < 0.5 else \
                    rnd.randrange(len(inflight))
                s, c = inflight.pop(i)
                holds[s] = c
                full[s].done += 1
        else:                       # a consumer stream
            c = nxt[actor]
            if c < pages:
                s = c % stages
                if full[s].test((c // stages) & 1):
                    if holds[s] != c:
                        return f"stream {actor} took stage {s} for page {c}, " \
                               f"which holds {holds[s]}"
                    empty[s].done += 1
                    nxt[actor] += nstream
    return "no progress"


@pytest.mark.parametrize("stages,nstream", [(8, 4), (16, 4), (4, 4), (8, 2),
                                            (16, 2), (4, 2)])
def test_ring_depth_multiple_of_streams_is_safe(stages, nstream):
    for seed in range(300):
        assert run(seed, stages, nstream) is None


def test_ring_depth_not_a_multiple_passes_early():
    """6 stages over 4 streams: some interleaving lets a stream consume a
    stage before its page has landed."""
    assert any(run(seed, 6, 4) is not None for seed in range(300))
