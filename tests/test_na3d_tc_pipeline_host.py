"""A CPU model of the tensor-core attention kernel's hand-over protocol
(rope_rope3d_apply_gb300/csrc/rope3d_na3d.cu, rope3d_na3d_tc_kernel).

The roles of one persistent CTA walking several query blocks are modelled:
  - the two TMA threads (K; V);
  - the two MMA threads (S products; P V products);
  - the Q warps, which have each block's Q tile copied by TMA (and rotate it
    in place in the rotating modes), store each block's O through the block's
    spent Q buffer and a TMA store and, in the mode that rotates K per CTA,
    rotate the K tiles;
  - the softmax threads, which write P over S in the S buffer.
Each role is a sequence of the kernel's mbarrier waits, arrivals and buffer
accesses. They run in many random interleavings over model mbarriers (a phase
counter, a pending arrival count and a transaction byte count each). The
layouts built are the kernel's: three S buffers with one O buffer (the
default), and two S buffers with two O buffers.

It asserts, in every interleaving, that:
  - every role runs to its end (no wait that can never be satisfied);
  - a wait on parity P is never made while the barrier is two or more phases
    past the phase it stands for (a parity wait cannot tell those apart);
  - no ring slot, S buffer or O buffer is written while a reader of the
    previous contents may still be reading it, nor read before it is written:
      - K slot s is overwritten only after the S MMAs of its last chunk;
      - V slot s only after that chunk's P V;
      - S buffer b (where the softmax writes P over S) only after the P V of
        the chunk one ring turn before has read its P;
      - O is rescaled only after the previous P V, and P V of chunk c runs on
        P and V of chunk c;
      - Q is rewritten only after the previous block's S MMAs;
      - a block's first P V overwrites an O buffer only after its previous
        block was read out of it, and row sums are read before rewritten.
The MMAs' completions are modelled as separate asynchronous events (a commit
arrives when the MMAs issued before it finish; each MMA thread's in order)."""
from __future__ import annotations

import random

import pytest


class Bar:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.phase = 0          # completed phases
        self.tx = 0

    def arrive(self):
        self.pending -= 1
        self._maybe_complete()

    def expect_tx(self, n):
        self.tx += n
        self.arrive()

    def complete_tx(self, n):
        self.tx -= n
        self._maybe_complete()

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def ready(self, parity, want_phase):
        """The kernel waits for parity (want_phase & 1) meaning 'phase
        want_phase has completed'; the wait is only sound if the barrier is
        at most one phase past it."""
        assert self.phase <= want_phase + 1, "parity wait outrun by two phases"
        assert parity == want_phase & 1
        return self.phase >= want_phase + 1


def simulate(blocks, rot_q, rot_k, seed, sbufs=3, drop_o_wait=False, drop=(), slow_q=False):
    """blocks: the chunk count of each query block the CTA walks in turn;
    sbufs: S buffers (3 with one O buffer, 2 with two)."""
    obufs = 1 if sbufs == 3 else 2
    rng = random.Random(seed)
    B = {}
    for s in (0, 1):   # K and V ring slots
        for kind, cnt in (("kFull", 1), ("kReady", 128), ("kEmpty", 1), ("vFull", 1), ("vEmpty", 1)):
            B[kind, s] = Bar(cnt)
    for b in range(sbufs):
        for kind, cnt in (("sFull", 1), ("sEmpty", 1), ("pFull", 256), ("pEmpty", 1)):
            B[kind, b] = Bar(cnt)
    for b in (0, 1):         # per Q buffer (block parity): Q landed (TMA), Q rotated, S MMAs done with it
        B["qFull", b], B["qReady", b], B["qEmpty", b] = Bar(1), Bar(128), Bar(1)
    for b in range(obufs):   # per O buffer: last P V done, O read out
        B["oReady", b], B["oEmpty", b] = Bar(1), Bar(128)
    for b in (0, 1):         # per block parity: row sums written
        B["oFull", b] = Bar(256)
    for b in (0, 1):         # per Q buffer: the TMA store of O staged in it has read it
        B["ostore", b] = Bar(1)
    for b in (0, 1):         # per block descriptor (block parity): written, read
        B["dFull", b], B["dEmpty", b] = Bar(128), Bar(256)
    B["qbar"] = Bar(4)       # the Q warps' named barrier (one arrival per modelled warp)
    for key, bar_ in B.items():   # planted mistakes: waits on these barriers are skipped
        bar_.dropped = (key[0] if isinstance(key, tuple) else key) in drop
    state = {  # what each buffer holds; S buffer b holds ("S", g) then ("P", g)
        "K": [None, None], "V": [None, None], "S": [None] * sbufs,
        "Q": [None, None],             # Q buffer: (block, "rot" or "raw") of the tile in it
        "O": [(-1, -1)] * obufs,       # O buffer: (block, last chunk added)
        "Oread": [-1] * obufs,         # O buffer: last block whose result was read out
        "sums": [-1, -1],              # row-sum buffer (block parity): block whose sums it holds
        "sums_read": [-1, -1],         # row-sum buffer: last block whose sums were read
        "pv_done": -1,                 # last chunk whose P V completed
        "s_done": -1,                  # last chunk whose S MMAs completed
        "staged": [0, 0],              # Q buffer: warps that wrote their O rows into it
        "desc": [None, None],          # descriptor slot: [block, softmax threads that read it]
    }
    inflight = []                      # asynchronous events: (kind, payload)
    SOFT = 4                           # softmax threads modelled (arrivals scaled)
    # global chunk g -> (block k, chunk c)
    seq = [(k, c) for k, n in enumerate(blocks) for c in range(n)]
    last_g = [sum(blocks[:k + 1]) - 1 for k in range(len(blocks))]

    def producer(kind):   # the K thread and the V thread, each over its own ring
        for g in range(len(seq)):
            s, use = g & 1, g >> 1
            if g >= 2:
                yield ("wait", B[kind + "Empty", s], (use - 1) & 1, use - 1)
            B[kind + "Full", s].expect_tx(2)
            inflight.append(("tma", (kind.upper(), s, g)))
            yield None

    def pv_issuer():
        for g, (k, c) in enumerate(seq):
            s, use = g & 1, g >> 1
            sb, suse = g % sbufs, g // sbufs
            ob = k % obufs
            if c == 0 and k >= obufs:   # O buffer ob read out by the Q warps (block k - obufs)
                u = k // obufs - 1
                yield ("wait", B["oEmpty", ob], u & 1, u)
            yield ("wait", B["pFull", sb], suse & 1, suse)
            yield ("wait", B["vFull", s], use & 1, use)
            assert state["S"][sb] == ("P", g) and state["V"][s] == g, "P V reads P and V of its chunk"
            if c == 0:   # the block's first P V overwrites O buffer ob
                assert state["Oread"][ob] == k - obufs or (k < obufs and state["Oread"][ob] == -1)
            inflight.append(("pv", (s, sb, g, k, c)))

    def s_issuer():
        for g, (k, c) in enumerate(seq):
            s, use = g & 1, g >> 1
            sb, suse = g % sbufs, g // sbufs
            if c == 0:
                yield ("wait", B["qReady" if rot_q else "qFull", k & 1], (k >> 1) & 1, k >> 1)
            yield ("wait", B["kReady" if rot_k else "kFull", s], use & 1, use)
            if g >= sbufs:
                yield ("wait", B["sEmpty", sb], (suse - 1) & 1, suse - 1)
            assert state["K"][s] == (g, "rot" if rot_k else "raw"), "S reads K of its chunk"
            assert state["Q"][k & 1] == (k, "rot" if rot_q else "raw"), "S reads Q of its block"
            inflight.append(("s", (s, sb, g, k, c == blocks[k] - 1)))

    def q_warp(i):
        g = 0
        ws = {"qb": 0, "ost": [0, 0], "ost_n": [0, 0], "pending": None}
        for k, n in enumerate(blocks):
            if k >= 2:                 # the softmax threads have read block k - 2's descriptor
                yield ("wait", B["dEmpty", k & 1], ((k - 2) >> 1) & 1, (k - 2) >> 1)
            if i == 0:
                d = state["desc"][k & 1]
                assert d is None or d == [k - 2, SOFT], "a descriptor is rewritten only after it was read"
                state["desc"][k & 1] = [k, 0]
            yield None                 # this warp's rows of the descriptor written
            for _ in range(32):
                B["dFull", k & 1].arrive()
            if k >= 2:                 # block k - 2's S MMAs are done with Q buffer k & 1
                yield ("wait", B["qEmpty", k & 1], ((k - 2) >> 1) & 1, (k - 2) >> 1)
            yield from o_reads_done(i, ws)   # and the TMA store of its O has read it
            if i == 0:                 # the tile by TMA into Q buffer k & 1
                B["qFull", k & 1].expect_tx(2)
                inflight.append(("tmaq", (k,)))
            yield None
            if rot_q:                  # landed, then rotated in place by every Q thread
                yield ("wait", B["qFull", k & 1], (k >> 1) & 1, k >> 1)
                assert state["Q"][k & 1] in ((k, "raw"), (k, "rot")), "the Q warps rotate their block's tile"
                yield None
                if i == 0:
                    state["Q"][k & 1] = (k, "rot")
                for _ in range(32):
                    B["qReady", k & 1].arrive()
            if k >= 1:                 # the previous block's result, before this block's K tiles
                yield from store_o(i, k - 1, ws)
            for c in range(n):         # K tiles: only the per-CTA mode has work here
                if rot_k:
                    s, use = g & 1, g >> 1
                    yield ("wait", B["kFull", s], use & 1, use)
                    if i == 0:
                        assert state["K"][s] == (g, "raw")
                        state["K"][s] = (g, "rot")
                    for _ in range(32):
                        B["kReady", s].arrive()
                    yield None
                g += 1
        yield from store_o(i, len(blocks) - 1, ws)
        if i == 0:                     # every store still out (a bulk-group wait), before the CTA ends
            for b in (0, 1):
                while ws["ost"][b] < ws["ost_n"][b]:
                    u = ws["ost"][b]
                    ws["ost"][b] += 1
                    yield ("wait", B["ostore", b], u & 1, u)

    def qbar(ws):                      # bar.sync among the four Q warps
        B["qbar"].arrive()
        n = ws["qb"]
        ws["qb"] += 1
        yield ("wait", B["qbar"], n & 1, n)

    def o_reads_done(i, ws):
        if ws["pending"] is not None:
            b = ws["pending"] & 1
            if i == 0:                 # the thread that committed the store waits for its reads
                u = ws["ost"][b]
                ws["ost"][b] += 1
                if not drop_o_wait:
                    yield ("wait", B["ostore", b], u & 1, u)
            yield from qbar(ws)
            ws["pending"] = None

    def store_o(i, k, ws):
        b, ob = k & 1, k % obufs
        u = k // obufs
        yield ("wait", B["oReady", ob], u & 1, u)
        yield ("wait", B["oFull", b], (k >> 1) & 1, k >> 1)
        assert state["O"][ob] == (k, blocks[k] - 1), "the block's O is complete"
        assert state["sums"][b] == k, "its row sums are written"
        # this warp's rows of O, normalised, into the block's own Q buffer
        assert state["s_done"] >= last_g[k], "the block's S MMAs no longer read its Q buffer"
        assert state["Q"][b] in ((k, "rot"), (k, "raw"), (k, "O")), "the Q buffer still holds block k"
        state["Q"][b] = (k, "O")
        state["staged"][b] += 1
        yield None
        if i == 0:
            state["Oread"][ob] = k
            state["sums_read"][b] = k
        for _ in range(32):
            B["oEmpty", ob].arrive()
        yield from qbar(ws)            # every warp's rows staged
        if i == 0:
            assert state["staged"][b] == 4, "the store reads all rows"
            inflight.append(("tmao", (k,)))
            ws["ost_n"][b] += 1
        ws["pending"] = k

    def softmax(i):
        g = 0
        for k, n in enumerate(blocks):
            m_valid = False
            ob = k % obufs
            yield ("wait", B["dFull", k & 1], (k >> 1) & 1, k >> 1)
            assert state["desc"][k & 1] is not None and state["desc"][k & 1][0] == k, \
                "the softmax reads its block's descriptor"
            state["desc"][k & 1][1] += 1
            for _ in range(256 // SOFT):
                B["dEmpty", k & 1].arrive()
            for c in range(n):
                sb, suse = g % sbufs, g // sbufs
                yield ("wait", B["sFull", sb], suse & 1, suse)
                assert state["S"][sb] in (("S", g), ("P", g)), "the softmax reads S of its chunk"
                yield None
                rescale = m_valid and rng.random() < 0.3
                m_valid = True
                # P(g) over S(g) in the same buffer (after the row's exchange)
                assert state["S"][sb] in (("S", g), ("P", g)), "S buffer still this chunk's"
                if i == 0:
                    state["S"][sb] = ("P", g)
                yield None
                if rescale:                    # after the weights are written
                    prev = g - 1
                    pb, pu = prev % sbufs, prev // sbufs
                    yield ("wait", B["pEmpty", pb], pu & 1, pu)
                    assert state["O"][ob] == (k, c - 1), "O rescaled after the previous P V"
                for _ in range(256 // SOFT):
                    B["pFull", sb].arrive()
                g += 1
                yield None
            # this part's row sums for the Q warps; on to the next block at once
            if i == 0:
                assert state["sums_read"][k & 1] == k - 2 or (k < 2 and state["sums_read"][k & 1] == -1), \
                    "row sums of block k - 2 were read"
                state["sums"][k & 1] = k
            for _ in range(256 // SOFT):
                B["oFull", k & 1].arrive()

    roles = [producer("k"), producer("v"), s_issuer(), pv_issuer()] + [softmax(i) for i in range(SOFT)] + \
        [q_warp(i) for i in range(4)]
    n_fast = len(roles) - 4   # the roles before the Q warps
    waiting = [None] * len(roles)
    done = [False] * len(roles)
    steps = 0
    while not all(done):
        steps += 1
        assert steps < 400000, "no progress"
        choices = [i for i in range(len(roles)) if not done[i]]
        runnable = [i for i in choices
                    if waiting[i] is None or waiting[i][0].ready(waiting[i][1], waiting[i][2])]
        if inflight and (not runnable or rng.random() < 0.4):
            kinds = [kd for kd, _ in inflight]
            if any(kd in ("tma", "tmao", "tmaq") for kd in kinds) and (
                    rng.random() < 0.5 or all(kd in ("tma", "tmao", "tmaq") for kd in kinds)):
                tma_idx = [j for j, kd in enumerate(kinds) if kd in ("tma", "tmao", "tmaq")]
                idx = rng.choice(tma_idx)
            else:   # each issuer's MMAs complete in its issue order
                first = [next((j for j, kd in enumerate(kinds) if kd == want), None) for want in ("s", "pv")]
                idx = rng.choice([j for j in first if j is not None])
            # a TMA store of a whole O tile takes long next to the Q warps' own
            # steps: it completes only now and then while anything else can move
            if kinds[idx] == "tmao" and runnable and rng.random() < 0.9:
                continue
            kind, pl = inflight.pop(idx)
            if kind == "tmaq":
                (kk,) = pl
                assert state["Q"][kk & 1] is None or state["Q"][kk & 1] == (kk - 2, "Oread"), \
                    "a Q buffer is rewritten only after the O staged in it was stored"
                state["Q"][kk & 1] = (kk, "raw")
                B["qFull", kk & 1].complete_tx(2)
            elif kind == "tmao":
                (kk,) = pl
                assert state["Q"][kk & 1] == (kk, "O") and state["staged"][kk & 1] == 4, \
                    "the store reads the staged O"
                state["Q"][kk & 1] = (kk, "Oread")
                state["staged"][kk & 1] = 0
                B["ostore", kk & 1].arrive()
            elif kind == "tma":
                buf, s, x = pl
                if buf == "K":
                    assert state["K"][s] is None or state["K"][s][0] <= x - 2
                    state["K"][s] = (x, "raw")
                    B["kFull", s].complete_tx(2)
                else:
                    assert state["V"][s] is None or state["V"][s] <= x - 2
                    state["V"][s] = x
                    B["vFull", s].complete_tx(2)
            elif kind == "s":
                s, sb, g, k, last = pl
                assert state["Q"][k & 1][0] == k, "Q kept until the block's S MMAs complete"
                # S(g) overwrites buffer sb only after P V of the chunk one ring
                # turn before has read the P in it
                assert state["S"][sb] is None or (state["S"][sb] == ("P", g - sbufs)
                                                  and state["pv_done"] >= g - sbufs)
                state["S"][sb] = ("S", g)
                state["s_done"] = g
                B["kEmpty", s].arrive()      # the commits after S(g)
                B["sFull", sb].arrive()
                if last:
                    B["qEmpty", k & 1].arrive()
            else:
                s, sb, g, k, c = pl
                ob = k % obufs
                prev = state["O"][ob]
                assert (c == 0) or prev == (k, c - 1), "P V in chunk order within the block"
                state["O"][ob] = (k, c)
                assert state["S"][sb] == ("P", g), "P kept until its P V completes"
                state["pv_done"] = g
                B["vEmpty", s].arrive()      # the commits after P V(g)
                B["pEmpty", sb].arrive()
                B["sEmpty", sb].arrive()     # S buffer sb free again
                if c == blocks[k] - 1:
                    B["oReady", ob].arrive()
            continue
        assert runnable, "deadlock"
        i = rng.choice(runnable)
        if slow_q and i >= n_fast and rng.random() < 0.9:   # the Q warps run rarely
            fast = [j for j in runnable if j < n_fast]
            if fast:
                i = rng.choice(fast)
        waiting[i] = None
        try:
            ev = next(roles[i])
            if ev is not None:
                _, bar, parity, phase = ev
                if not bar.dropped:
                    waiting[i] = (bar, parity, phase)
        except StopIteration:
            done[i] = True
    assert not inflight
    assert state["pv_done"] == len(seq) - 1


BLOCKS = [[1], [3], [8], [1, 1, 1], [3, 2, 4], [8, 8, 6, 8], [2, 5, 1, 7, 3], [1, 2, 1, 2, 1]]


@pytest.mark.parametrize("sbufs", [3, 2])
@pytest.mark.parametrize("blocks", BLOCKS, ids=[str(b) for b in BLOCKS])
@pytest.mark.parametrize("mode", ["none", "q", "qk"])
def test_pipeline_protocol(blocks, mode, sbufs):
    for seed in range(40):
        simulate(blocks, mode != "none", mode == "qk", seed * 7919 + len(blocks), sbufs)


@pytest.mark.parametrize("blocks", [[3, 2, 4], [8, 8, 6, 8]], ids=str)
def test_protocol_model_catches_a_dropped_wait(blocks):
    """A planted mistake: the Q warps copy the next Q tile into a buffer
    without waiting for the TMA store of the O staged there to have read it.
    Some interleaving must then find the buffer overwritten under the store."""
    messages = set()
    for seed in range(40):
        try:
            simulate(blocks, True, False, seed, 3, drop_o_wait=True)
        except AssertionError as e:
            messages.add(str(e).split("\n")[0])
    assert any("staged" in m_ for m_ in messages), messages


@pytest.mark.parametrize("wait", ["sEmpty", "oEmpty", "kEmpty", "vEmpty", "dFull", "sFull", "pFull", "oFull"])
def test_protocol_model_catches_each_dropped_wait(wait):
    """Planted mistakes: every wait on one kind of barrier skipped. Some
    interleaving (the Q warps running slowly in half of them) must then fail
    one of the model's assertions."""
    failed = 0
    for seed in range(40):
        try:
            simulate([3, 2, 4, 1, 2], True, False, seed, 3, drop=(wait,), slow_q=seed % 2 == 1)
        except AssertionError:
            failed += 1
    assert failed > 0


@pytest.mark.parametrize("wait", ["dEmpty", "qEmpty"])
def test_protocol_waits_implied_by_the_o_hand_over(wait):
    """Two waits of the Q warps are implied by an earlier one: before block
    k's descriptor and Q tile go into slot and buffer k & 1, the Q warps have
    stored block k - 2's O, which waited for its last P V (after all its S
    products) and for all its softmax row sums (after every softmax thread read
    its descriptor). Dropping either changes nothing, even with slow Q warps."""
    for seed in range(40):
        simulate([3, 2, 4, 1, 2], True, False, seed, 3, drop=(wait,), slow_q=seed % 2 == 1)
