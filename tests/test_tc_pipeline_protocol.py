"""A model of the tcgen05 attention kernel's barrier protocol, run under
random interleavings on the CPU.

The kernel (attention_tc.cu) is a pipeline of a producer warp (TMA copies
of K+V tiles into a ring and of each segment's Q), one MMA-issuing thread,
and two softmax groups of four warps, synchronised by mbarriers with
parity waits.  A parity wait cannot tell phase k from phase k + 2, so a
waiter must never fall two phases behind a barrier; and every wait must be
able to end.  This model replays the same protocol -- barrier counts, the
order of arrivals and waits, which side waits for what -- with:

* TMA copies that land in any order;
* MMAs that complete in issue order, and commits (tcgen05.commit) that
  arrive in any order once every MMA issued before them has completed;
* any interleaving of the producer, the MMA thread and the eight softmax
  warps.

It checks that every run completes, that no wait sees a lapped phase, and
that every buffer read sees the data of the tile it is meant for (the K/V
stage, Q of the segment, the S and O accumulators, the P buffer).  Both
modes are modelled:

* one row group per tile: two groups on alternate tiles, three stages, P in
  a buffer per group, state handed from group 1 to group 0 at a segment's
  end;
* two row groups: both groups on every tile, three stages, one S MMA per
  tile for both groups into a double-buffered S with one barrier per S
  buffer parity, each group's P written into the stage's K tile (free once
  the S MMA has completed) as rows of one operand shared by both groups, a
  segment's output staged there too (over both groups' P); one P V per
  tile for both groups, issued once both groups' P are written, followed
  by a commit to each group's O barrier and, except on a segment's last
  tile, two commits to the stage's empty barrier; a segment's last stage
  goes back to the producer on each group's own arrival once its staged
  output has been read.

Controls show the model finds the hazards the kernel avoids: a single S
barrier for all tiles (instead of one per parity) laps, separate S MMAs
with a commit each let a group overwrite K while the other group's S MMA
still reads it, releasing a segment's last stage right after its P V lets
the producer overwrite the staged output, issuing the shared P V once one
group's P is written reads the other group's rows before they are (or its
O before it is folded), and
issuing Q only when its release has been seen (without waiting for it
before blocking on a stage of the same segment) deadlocks.
"""
import random

import pytest


class Lap(Exception):
    pass


class Stuck(Exception):
    pass


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pend, self.done = name, count, 0, 0

    def arrive(self):
        self.pend += 1
        assert self.pend <= self.count, self.name
        if self.pend == self.count:
            self.pend = 0
            self.done += 1

    def test(self, parity):
        return (self.done & 1) != parity


def wait(bar, k):
    """Wait for phase k (parity k & 1); a lapped phase is an error."""
    while True:
        if bar.done > k + 1:
            raise Lap(f"{bar.name}: waited for phase {k}, {bar.done} done")
        if bar.test(k & 1):
            return
        yield


class Hazard(Exception):
    pass


def run(seed, dual, single_s_barrier=False, lazy_q_only=False, R=4,
        separate_s_commits=False, early_release=False, pv_on_one_p=False):
    rnd = random.Random(seed)
    ST = 3
    segs = [rnd.randint(1, 7) for _ in range(rnd.randint(1, 6))]
    full = [Bar(f"full{s}", 1) for s in range(ST)]
    empty = [Bar(f"empty{s}", 2 if dual else 1) for s in range(ST)]
    n_s = 1 if single_s_barrier else 4 if separate_s_commits else 2
    s_full = [Bar(f"s_full{i}", 1) for i in range(n_s)]
    p_full = [Bar(f"p_full{g}", 4) for g in range(2)]
    o_full = [Bar(f"o_full{g}", 1) for g in range(2)]
    q_full, q_empty = Bar("q_full", 1), Bar("q_empty", 1)
    ufull = [Bar(f"ufull{u}", 1) for u in range(R)]
    uempty = [Bar(f"uempty{u}", 3) for u in range(R)]
    x_full = [Bar(f"x_full{k}", 4) for k in range(2)]
    x_empty = [Bar(f"x_empty{k}", 4) for k in range(2)]
    stg_free = Bar("stg_free", 1)

    unit = [None] * R
    stage = [None] * ST      # tile whose K/V a stage holds
    # two row groups: what each group's part of a stage's K tile holds
    # ("K" until a group writes P there, then ("P", tile), ("out", seg))
    kpart = [[None, None] for _ in range(ST)]
    qbuf = [None]            # segment whose Q is in the Q buffer
    seg_of = {}              # tile -> segment
    sbuf, obuf, pbuf = {}, [None, None], [None, None]
    copies = []              # (barrier, setter) in flight
    pipe = []                # issued MMAs and commits, in issue order
    commits = []             # commits whose MMAs are all complete

    def s_bar(g, c):
        if dual:
            if single_s_barrier:
                return s_full[0], c
            if separate_s_commits:   # one barrier per group and S buffer
                return s_full[2 * g + (c & 1)], c >> 1
            return s_full[c & 1], c >> 1
        return s_full[g], c >> 1

    def o_phase(t):
        return t if dual else t >> 1

    def land(s, c):
        if dual and "out" in [k[0] if k else None for k in kpart[s]]:
            raise Hazard(f"copy into stage {s} over a staged output")
        stage[s] = c
        kpart[s] = ["K", "K"]

    def copy_engine():
        while True:
            if copies and rnd.random() < 0.5:
                bar, setter = copies.pop(rnd.randrange(len(copies)))
                setter()
                bar.arrive()
            yield

    def tensor_core():
        while True:
            if pipe and pipe[0][0] != "commit" and rnd.random() < 0.5:
                op = pipe.pop(0)
                kind, g, c = op
                s = c % ST
                assert stage[s] == c, ("MMA reads stage", stage[s], c)
                if kind == "S":
                    assert qbuf[0] == seg_of[c], ("S reads Q", qbuf[0], seg_of[c])
                    if dual and kpart[s] != ["K", "K"]:
                        raise Hazard(f"S({c}) reads K overwritten: {kpart[s]}")
                    for gg in ((0, 1) if g is None else (g,)):
                        sbuf[(gg, c & 1) if dual else gg] = c
                elif g is None:  # both groups' P V: one operand of both P
                    if kpart[s] != [("P", c), ("P", c)]:
                        raise Hazard(f"P V({c}) reads {kpart[s]}")
                    obuf[0] = obuf[1] = c
                else:
                    assert pbuf[g] == c, ("P V reads P", pbuf[g], c)
                    obuf[g] = c
            while pipe and pipe[0][0] == "commit":
                commits.append(pipe.pop(0)[1])
            if commits and rnd.random() < 0.5:
                commits.pop(rnd.randrange(len(commits))).arrive()
            yield

    def producer():
        c = 0
        for us, nt in enumerate(segs + [None]):
            slot = us % R
            if us >= R:
                yield from wait(uempty[slot], us // R - 1)
            unit[slot] = nt
            ufull[slot].arrive()
            if nt is None:
                return
            q_pending, seg_c0 = True, c

            def issue_q(u=us):
                copies.append((q_full, lambda: qbuf.__setitem__(0, u)))

            for _ in range(nt):
                if q_pending:
                    must = c - ST >= seg_c0 and not lazy_q_only
                    if must and us > 0:
                        yield from wait(q_empty, us - 1)
                    if us == 0 or q_empty.done >= us:
                        issue_q()
                        q_pending = False
                s = c % ST
                if c >= ST:
                    yield from wait(empty[s], c // ST - 1)
                seg_of[c] = us
                copies.append((full[s], lambda s=s, c=c: land(s, c)))
                c += 1
                yield
            if q_pending:
                if us > 0:
                    yield from wait(q_empty, us - 1)
                issue_q()

    def mma():
        c_s = us = left = 0
        first = no_more = False
        c_p, p_obs = [0, 0], [0, 0]   # alternating mode uses index 0
        last_tiles = set()            # tiles that end a segment
        while True:
            if left == 0 and not no_more and ufull[us % R].test((us // R) & 1):
                nt = unit[us % R]
                uempty[us % R].arrive()
                us += 1
                if nt is None:
                    no_more = True
                else:
                    left, first = nt, True
            ready = (p_obs[0] >= c_s - 1 and p_obs[1] >= c_s - 1) if dual \
                else p_obs[0] >= c_s - 1
            if (left > 0 and ready and full[c_s % ST].test((c_s // ST) & 1)
                    and (not first or q_full.test((us - 1) & 1))):
                if dual and separate_s_commits:
                    for g in (0, 1):
                        pipe.append(("S", g, c_s))
                        pipe.append(("commit", s_bar(g, c_s)[0]))
                elif dual:
                    pipe.append(("S", None, c_s))
                    pipe.append(("commit", s_bar(0, c_s)[0]))
                else:
                    g = c_s & 1
                    pipe.append(("S", g, c_s))
                    pipe.append(("commit", s_bar(g, c_s)[0]))
                c_s += 1
                left -= 1
                first = False
                if left == 0:
                    pipe.append(("commit", q_empty))
                    last_tiles.add(c_s - 1)
            if dual:
                for g in (0, 1):
                    if p_obs[g] < c_s and p_full[g].test(p_obs[g] & 1):
                        p_obs[g] += 1
                if c_p[0] < p_obs[0] and (pv_on_one_p or c_p[0] < p_obs[1]):
                    c = c_p[0]
                    pipe.append(("PV", None, c))
                    pipe.append(("commit", o_full[0]))
                    pipe.append(("commit", o_full[1]))
                    c_p[0] += 1
                    # a segment's last stage goes back from the groups, once
                    # their staged outputs were read
                    if c not in last_tiles or early_release:
                        pipe.append(("commit", empty[c % ST]))
                        pipe.append(("commit", empty[c % ST]))
                if no_more and left == 0 and c_p[0] == c_s:
                    return
            else:
                k = p_obs[0]
                if k < c_s and p_full[k & 1].test((k >> 1) & 1):
                    p_obs[0] += 1
                if c_p[0] < p_obs[0]:
                    c = c_p[0]
                    pipe.append(("PV", c & 1, c))
                    pipe.append(("commit", empty[c % ST]))
                    pipe.append(("commit", o_full[c & 1]))
                    c_p[0] += 1
                if no_more and left == 0 and c_p[0] == c_s:
                    return
            yield

    def warp(g, w):
        c0 = us = 0
        while True:
            slot = us % R
            yield from wait(ufull[slot], us // R)
            nt = unit[slot]
            if nt is None:
                return
            prev = -1
            taus = range(nt) if dual else range(0 if (c0 & 1) == g else 1, nt, 2)
            for tau in taus:
                c = c0 + tau
                bar, k = s_bar(g, c)
                yield from wait(bar, k)
                yield from wait(full[c % ST], c // ST)
                assert sbuf[(g, c & 1) if dual else g] == c, ("S", c)
                assert stage[c % ST] == c, ("V rows cleared", stage[c % ST], c)
                yield
                if prev >= 0:
                    yield from wait(o_full[g], o_phase(prev))
                    assert obuf[g] == prev, ("fold O", obuf[g], prev)
                if not dual and g == 1 and prev < 0 and us > 0:
                    yield from wait(stg_free, us - 1)
                if dual:
                    kpart[c % ST][g] = ("P", c)
                else:
                    pbuf[g] = c
                p_full[g].arrive()
                prev = c
                yield
            if prev >= 0:
                yield from wait(o_full[g], o_phase(prev))
                assert obuf[g] == prev
            if dual:
                # the group's output is staged in the last tile's K (over
                # rows of both groups' P), read by the bulk stores, then
                # released
                s = prev % ST
                if w == 0:
                    if stage[s] != prev:
                        raise Hazard(f"staging in stage {s} now holding {stage[s]}")
                    kpart[s][g] = ("out", us)
                    kpart[s][1 - g] = ("out", us) if kpart[s][1 - g] == ("P", prev) \
                        else kpart[s][1 - g]
                    yield
                    if kpart[s][g] != ("out", us) or stage[s] != prev:
                        raise Hazard(f"staged output of segment {us} overwritten")
                    kpart[s][g] = ("done", us)
                    if not early_release:
                        empty[s].arrive()
            else:
                xk = us & 1
                if g == 1:
                    if us >= 2:
                        yield from wait(x_empty[xk], (us >> 1) - 1)
                    x_full[xk].arrive()
                else:
                    yield from wait(x_full[xk], us >> 1)
                    x_empty[xk].arrive()
                    if w == 0:
                        stg_free.arrive()
            if w == 0:
                uempty[slot].arrive()
            c0 += nt
            us += 1

    agents = {"producer": producer(), "mma": mma(), "copy": copy_engine(),
              "tc": tensor_core()}
    for g in (0, 1):
        for w in range(4):
            agents[f"g{g}w{w}"] = warp(g, w)
    finite = [k for k in agents if k not in ("copy", "tc")]
    done = set()
    for _ in range(200_000):
        if len(done) == len(finite):
            return
        k = rnd.choice([k for k in agents if k not in done])
        try:
            next(agents[k])
        except StopIteration:
            done.add(k)
    raise Stuck(f"no progress: finished {sorted(done)}, segments {segs}")


@pytest.mark.parametrize("dual", [False, True], ids=["one-row-group", "two-row-groups"])
def test_protocol_completes_without_laps_or_hazards(dual):
    for seed in range(400):
        run(seed, dual)


def test_one_s_barrier_for_all_tiles_laps_with_two_row_groups():
    """Control: with double-buffered S and a single S barrier (instead of
    one per buffer parity), S(c + 1) can complete before a group has waited
    for S(c)."""
    failures = 0
    for seed in range(200):
        try:
            run(seed, True, single_s_barrier=True)
        except (Lap, Stuck):
            failures += 1
    assert failures > 0


def test_separate_s_commits_let_p_overwrite_k_in_use():
    """Control: with a commit after each group's S MMA, a group can see its
    own S complete and write P into the stage's K tile while the other
    group's S MMA still reads it."""
    failures = 0
    for seed in range(400):
        try:
            run(seed, True, separate_s_commits=True)
        except Hazard:
            failures += 1
    assert failures > 0


def test_releasing_a_segments_last_stage_early_overwrites_its_output():
    """Control: handing a segment's last stage back right after its P V lets
    the producer copy the next tile over the output staged there."""
    failures = 0
    for seed in range(400):
        try:
            run(seed, True, early_release=True)
        except Hazard:
            failures += 1
    assert failures > 0


def test_shared_p_v_issued_on_one_groups_p_reads_unwritten_rows():
    """Control: the P V that serves both groups issued as soon as group 0's
    P is written reads group 1's rows before group 1 has written them, or
    overwrites group 1's O before group 1 has folded it (its O barrier then
    laps, or its arrivals run ahead of its waits)."""
    failures = 0
    for seed in range(400):
        try:
            run(seed, True, pv_on_one_p=True)
        except (Hazard, AssertionError, Lap, Stuck):
            failures += 1
    assert failures > 0


@pytest.mark.parametrize("dual", [False, True], ids=["one-row-group", "two-row-groups"])
def test_q_issued_only_on_a_seen_release_can_deadlock(dual):
    """Control: the producer issues a segment's Q only if the old Q's
    release has been seen; blocking on a stage whose previous tile is of the
    same segment then waits for an S that needs that Q.  Commits need not
    arrive in issue order, so the release can still be pending there."""
    failures = 0
    for seed in range(400):
        try:
            run(seed, dual, lazy_q_only=True)
        except Stuck:
            failures += 1
    assert failures > 0
