"""A CPU model of the tensor-core decode kernel's four warp roles and their
mbarriers (CPU only; no GPU involved).

The kernel (decode_kv_cache_gb300/csrc/lf_decode_tc.cuh) runs, in every CTA,
a producer warp (TMA tiles into a ring of S stages), an MMA warp, four
epilogue warps and two tail warps.  They hand work to each other only through
mbarriers: the tile ring (full / empty), the logit accumulators (sfull /
sfree, 16 of them), the P^T tiles (pready / pfree, 4), the output accumulator
(ofull), and the per-parity unit buffers (aux / auxfree, statrdy, handoff,
taildone).  The ring order is shared by the producer and the MMA warp: K of
the first non-empty unit, then for each next non-empty unit its first L K
tiles, the V tiles of the unit before it, and its remaining K tiles.  A V
block still pending when the walk reaches two units past it is issued alone
first (the flush), because the producer's wait on the unit-2 buffers needs it.

Here each role is a generator that performs the same arrivals and waits in the
same order as its warp; a random scheduler interleaves them.  The model checks,
over many seeded patterns of empty and non-empty units:
  * liveness: every role finishes (no state where all remaining roles wait);
  * no phase aliasing: a parity wait never sees its barrier two or more phases
    past the phase it waits for (the hardware wait would then block or pass on
    the wrong phase);
  * the producer's ring order and the MMA warp's are the same tile for tile.
Planting a mistake shows the checks bite: without the flush the model finds
deadlocks (the epilogue waits for a unit's output whose V tiles the producer
holds back), and a flush in the producer alone breaks the shared order.
ClusterModel adds the exchanges between the CTAs of a cluster (clusters of 1,
2 and 4; each CTA holds its share of every unit, possibly none): every CTA's
(m, l) to every CTA, then its partial output to the unit's leader.  Each
transfer checks that it lands in the phase it is meant for and that the
receiving buffer is no longer read; a planted single statistics buffer fails
that check.  For planned launches the model puts a cluster's part of a shared
unit first, exchanged through global memory (taken as immediate here: the
other clusters are not modelled, and a shared unit uses neither the
statistics receive buffers nor their barriers), and checks the whole units'
corrected phase indices.
"""
import random

import pytest

SBUFS, PBUFS = 16, 4     # logit accumulators and P^T tiles in flight (as in the kernel)
TILE = 128


def ntiles(rows):
    return (rows + TILE - 1) // TILE


def ring_order(rows, lookahead, flush):
    """The tile order one role derives from the unit list: (kind, item, tile)."""
    order, prev = [], None
    for k, r in enumerate(rows):
        if flush and prev is not None and prev <= k - 2:
            order += [("V", prev, t) for t in range(ntiles(rows[prev]))]
            prev = None
        if r == 0:
            continue
        nt = ntiles(r)
        if prev is None:
            order += [("K", k, t) for t in range(nt)]
        else:
            L = min(nt, lookahead)
            order += [("K", k, t) for t in range(L)]
            order += [("V", prev, t) for t in range(ntiles(rows[prev]))]
            order += [("K", k, t) for t in range(L, nt)]
        prev = k
    if prev is not None:
        order += [("V", prev, t) for t in range(ntiles(rows[prev]))]
    return order


class Model:
    def __init__(self, rows, stages, lookahead, producer_flush=True, mma_flush=True,
                 cta=0, count=None):
        self.rows = rows
        self.S = stages
        self.L = lookahead
        self.cta = cta
        self.count = {} if count is None else count   # (cta, barrier, slot) -> completed phases
        self.produced = []       # ring order as issued by the producer
        self.consumed = []       # ring order as consumed by the MMA warp
        self.pflush, self.mflush = producer_flush, mma_flush

    # -- barriers -------------------------------------------------------------
    def arrive(self, name, slot=0):
        key = (self.cta, name, slot)
        self.count[key] = self.count.get(key, 0) + 1

    def done(self, wait):
        name, slot, phase = wait
        c = self.count.get((self.cta, name, slot), 0)
        assert c <= phase + 1, f"phase aliasing on {name}[{slot}]: {c} completions, waits for {phase}"
        return c >= phase + 1

    # -- roles (same arrivals and waits, in the same order, as the warps) -------
    def producer(self):
        S, tt = self.S, 0
        order = ring_order(self.rows, self.L, self.pflush)
        # split the order at the points where the producer handles each item
        prev = None
        plan = []                 # (item, tiles to flush first, tiles of the item)
        o = 0
        for k, r in enumerate(self.rows):
            flush = []
            if self.pflush and prev is not None and prev <= k - 2:
                n = ntiles(self.rows[prev])
                flush = order[o:o + n]
                o += n
                prev = None
            own = []
            if r > 0:
                n = ntiles(r) + (ntiles(self.rows[prev]) if prev is not None else 0)
                own = order[o:o + n]
                o += n
                prev = k
            plan.append((k, flush, own))
        tail = order[o:]

        def emit(tiles):
            nonlocal tt
            for tile in tiles:
                if tt >= S:
                    yield ("empty", tt % S, tt // S - 1)
                self.produced.append(tile)
                self.arrive("full", tt % S)       # the TMA bytes land
                tt += 1

        for k, flush, own in plan:
            yield from emit(flush)
            if k >= 2:
                yield ("auxfree", k & 1, (k >> 1) - 1)
            self.arrive("aux", k & 1)             # ||v|| and positions of unit k
            yield from emit(own)
        yield from emit(tail)

    def mma(self):
        S = self.S
        order = ring_order(self.rows, self.L, self.mflush)
        tt = kt = pt = 0
        for tile in order:
            kind = tile[0]
            if kind == "K":
                yield ("full", tt % S, tt // S)
                if kt >= SBUFS:
                    yield ("sfree", kt % SBUFS, kt // SBUFS - 1)
                self.consumed.append(tile)
                self.arrive("sfull", kt % SBUFS)
                self.arrive("empty", tt % S)
                kt += 1
            else:
                yield ("pready", pt % PBUFS, pt // PBUFS)
                yield ("full", tt % S, tt // S)
                self.consumed.append(tile)
                self.arrive("empty", tt % S)
                self.arrive("pfree", pt % PBUFS)
                pt += 1
                item, t = tile[1], tile[2]
                if t == ntiles(self.rows[item]) - 1:
                    self.arrive("ofull")          # the unit's output accumulator is final
            tt += 1

    def epilogue(self):
        kt = pt = ne = 0
        for k, r in enumerate(self.rows):
            if k >= 2:
                yield ("taildone", k & 1, (k >> 1) - 1)
            yield ("aux", k & 1, k >> 1)
            for _ in range(ntiles(r)):
                yield ("sfull", kt % SBUFS, kt // SBUFS)
                self.arrive("sfree", kt % SBUFS)
                kt += 1
            self.arrive("auxfree", k & 1)
            if r > 0:
                for _ in range(ntiles(r)):
                    if pt >= PBUFS:
                        yield ("pfree", pt % PBUFS, pt // PBUFS - 1)
                    self.arrive("pready", pt % PBUFS)
                    pt += 1
                self.arrive("statrdy", k & 1)
                yield ("ofull", 0, ne)
                ne += 1
            else:
                self.arrive("statrdy", k & 1)
            self.arrive("handoff", k & 1)

    def tail(self):
        for k in range(len(self.rows)):
            yield ("statrdy", k & 1, k >> 1)
            yield ("handoff", k & 1, k >> 1)
            self.arrive("taildone", k & 1)

    # -- a random interleaving ---------------------------------------------------
    def run(self, rng):
        roles = {"producer": self.producer(), "mma": self.mma(), "epilogue": self.epilogue(),
                 "tail": self.tail()}
        waits = {}
        for name, g in roles.items():
            w = next(g, None)
            if w is not None:
                waits[name] = w
        while waits:
            ready = [n for n, w in waits.items() if self.done(w)]
            if not ready:
                return "deadlock", dict(waits)
            n = rng.choice(ready)
            w = next(roles[n], None)
            if w is None:
                del waits[n]
            else:
                waits[n] = w
        return "done", None


class TxBarrier:
    """An mbarrier completed by its owner's arrive.expect_tx plus `senders`
    remote st.async transfers.  A transfer must land in the phase it is meant
    for: landing while the previous phase is still open would complete that one
    with the wrong data."""

    def __init__(self, senders):
        self.senders = senders
        self.completed = 0
        self.landed = 0
        self.armed = False

    def _maybe_complete(self):
        if self.armed and self.landed == self.senders:
            self.completed += 1
            self.landed, self.armed = 0, False

    def arm(self, phase):
        assert self.completed == phase and not self.armed, (self.completed, phase)
        self.armed = True
        self._maybe_complete()

    def land(self, phase):
        assert self.completed == phase, f"transfer for phase {phase} lands in phase {self.completed}"
        self.landed += 1
        assert self.landed <= self.senders
        self._maybe_complete()


class ClusterModel:
    """C CTAs of one cluster walk the same unit list; CTA `rank` holds the
    slots [rank*per, (rank+1)*per) of each unit (per = ceil(n/C) rounded up
    to 4).  Besides the roles of every CTA, the tail warps run the two
    exchanges: every CTA sends its (m, l) to every CTA (statb, one buffer per
    unit parity), then its partial output to the unit's leader, rank k mod C
    (finb, a single buffer).  Each transfer checks that the receiving buffer
    is free: the receiver has finished the unit that last used it."""

    def __init__(self, occupied, cluster, stages, lookahead, mistake=None, shared=0):
        self.n = occupied
        self.C = cluster
        self.mistake = mistake    # a planted protocol error (tests of the model itself)
        # planned launch: items 0 .. shared-1 are units shared with other clusters,
        # exchanged through global memory (modelled as immediate); they use neither
        # statb nor finb nor the statistics receive buffers
        self.shared = shared
        self.count = {}
        self.ctas = []
        for r in range(cluster):
            rows = []
            for n in occupied:
                per = ((n + cluster - 1) // cluster + 3) & ~3
                rows.append(max(0, min(per, n - r * per)))
            m = Model(rows, stages, lookahead, cta=r, count=self.count)
            m.tail = self._tail_fn(m)
            self.ctas.append(m)
        self.statb = {(r, b): TxBarrier(cluster) for r in range(cluster) for b in (0, 1)}
        self.finb = {r: TxBarrier(cluster) for r in range(cluster)}
        self.stats_read = [-1] * cluster   # last unit whose statistics each CTA has read
        self.tail_done = [0] * cluster     # units each CTA's tail has finished

    def _tail_fn(self, m):
        C, r = self.C, m.cta

        def tail():
            for k in range(len(self.n)):
                b2 = k & 1
                yield ("statrdy", b2, k >> 1)
                if k < self.shared:
                    yield ("handoff", b2, k >> 1)
                    self.tail_done[r] += 1
                    m.arrive("taildone", b2)
                    continue
                # the shared items completed no statb / finb phase: the phase index of
                # a whole unit counts only the whole units before it
                npc = self.shared if self.mistake != "uncorrected_phases" else 0
                # exchange 1: arm this parity's receive barrier, send (m, l) to all
                if self.mistake == "one_statistics_buffer":
                    sb, sp, prev = 0, k, k - 1      # (planted) one buffer for every unit
                else:
                    k0 = npc + ((k - npc) & 1)     # first whole item of this parity
                    sb, sp, prev = b2, (k - k0) >> 1, k - 2
                self.statb[(r, sb)].arm(sp)
                for dst in range(C):
                    # the buffer's previous user (a whole unit) has been read at dst
                    assert prev < self.shared or self.stats_read[dst] >= prev, \
                        "statistics buffer still in use"
                    self.statb[(dst, sb)].land(sp)
                yield ("statb", sb, sp)
                self.stats_read[r] = k
                yield ("handoff", b2, k >> 1)          # the partial output is read
                # exchange 2: partial output and lowest candidate to the leader
                leader = (k - npc) % C
                fp = (k - npc) // C
                if r == leader:
                    self.finb[r].arm(fp)
                assert k - npc < C or self.tail_done[leader] >= k - C + 1, \
                    "output buffer still in use"
                self.finb[leader].land(fp)
                if r == leader:
                    yield ("finb", 0, fp)
                self.tail_done[r] += 1
                m.arrive("taildone", b2)
        return tail

    def done(self, cta, wait):
        name, slot, phase = wait
        if name == "statb":
            bar = self.statb[(cta, slot)]
        elif name == "finb":
            bar = self.finb[cta]
        else:
            return self.ctas[cta].done(wait)
        assert bar.completed <= phase + 1
        return bar.completed >= phase + 1

    def run(self, rng):
        roles = {}
        for m in self.ctas:
            for name, fn in (("producer", m.producer), ("mma", m.mma), ("epilogue", m.epilogue),
                             ("tail", m.tail)):
                roles[(m.cta, name)] = fn()
        waits = {}
        for key, g in roles.items():
            w = next(g, None)
            if w is not None:
                waits[key] = w
        while waits:
            ready = [key for key, w in waits.items() if self.done(key[0], w)]
            if not ready:
                return "deadlock", dict(waits)
            key = rng.choice(ready)
            w = next(roles[key], None)
            if w is None:
                del waits[key]
            else:
                waits[key] = w
        return "done", None


def random_rows(rng, n_items):
    rows = []
    for _ in range(n_items):
        x = rng.random()
        if x < 0.4:
            rows.append(0)                               # empty: no share of this unit here
        elif x < 0.6:
            rows.append(rng.randint(1, TILE))            # one (ragged) tile
        else:
            rows.append(rng.randint(TILE + 1, 14 * TILE))
    return rows


@pytest.mark.parametrize("stages,lookahead", [(3, 2), (2, 1), (4, 3), (3, 8)])
def test_kernel_protocol_is_live_and_alias_free(stages, lookahead):
    rng = random.Random(1000 * stages + lookahead)
    for trial in range(400):
        rows = random_rows(rng, rng.randint(1, 12))
        m = Model(rows, stages, lookahead)
        status, waits = m.run(rng)
        assert status == "done", (rows, waits)
        assert m.produced == m.consumed == ring_order(rows, lookahead, True)
        assert all(m.count.get((0, "handoff", b), 0) == (len(rows) + 1 - b) // 2 for b in (0, 1))


def test_without_the_flush_a_unit_after_two_empty_ones_deadlocks():
    rows = [300, 0, 0, 200]
    status, waits = Model(rows, 3, 2, producer_flush=False, mma_flush=False).run(random.Random(0))
    assert status == "deadlock"
    # the epilogue waits for unit 0's output; the producer holds its V tiles back
    assert waits["epilogue"][0] == "ofull" and waits["producer"][0] == "auxfree"
    assert Model(rows, 3, 2).run(random.Random(0))[0] == "done"


def test_without_the_flush_random_patterns_deadlock():
    rng = random.Random(7)
    found = 0
    for _ in range(300):
        rows = random_rows(rng, rng.randint(3, 12))
        if Model(rows, 3, 2, producer_flush=False, mma_flush=False).run(rng)[0] == "deadlock":
            found += 1
    assert found > 0      # 115 of these 300 patterns


def test_flush_in_one_role_only_breaks_the_shared_order():
    rows = [300, 0, 0, 200]
    m = Model(rows, 3, 2, producer_flush=True, mma_flush=False)
    status, _ = m.run(random.Random(0))
    # the MMA warp reads a stage as the wrong tile (here: a V tile of unit 0 as K of unit 3)
    assert any(p != c for p, c in zip(m.produced, m.consumed)) or status == "deadlock"


@pytest.mark.parametrize("cluster", [1, 2, 4])
def test_cluster_exchanges_are_live_and_reuse_free_buffers(cluster):
    """Units of every size, including ones that leave some CTAs of the cluster
    without slots (fewer than C*4 occupied), under random interleavings of all
    roles of all CTAs."""
    rng = random.Random(31 + cluster)
    for _ in range(250):
        occupied = []
        for _ in range(rng.randint(1, 10)):
            x = rng.random()
            occupied.append(0 if x < 0.15 else rng.randint(1, 4 * cluster) if x < 0.4
                            else rng.randint(1, 3276))
        m = ClusterModel(occupied, cluster, 3, 2)
        status, waits = m.run(rng)
        assert status == "done", (occupied, waits)
        assert m.tail_done == [len(occupied)] * cluster
        for c in m.ctas:
            assert c.produced == c.consumed


def test_cluster_model_catches_a_single_statistics_buffer():
    """Planted: one statistics receive buffer instead of one per unit parity.
    A CTA that has finished a unit's first exchange can then send the next
    unit's statistics while a slower peer is still reading the previous ones."""
    rng = random.Random(5)
    caught = 0
    for _ in range(200):
        occupied = [rng.randint(1, 3276) for _ in range(rng.randint(3, 10))]
        try:
            ClusterModel(occupied, 2, 3, 2, mistake="one_statistics_buffer").run(rng)
        except AssertionError as e:
            assert "statistics buffer still in use" in str(e)
            caught += 1
    assert caught > 0


@pytest.mark.parametrize("cluster,shared", [(1, 1), (2, 1), (4, 1), (2, 2)])
def test_planned_launch_phase_indices(cluster, shared):
    """Planned launches put a cluster's part of a shared unit first; it is
    exchanged through global memory, so it completes no statb / finb phase
    and uses no statistics receive buffer.  The whole units' phase indices
    and leaders count only the whole units (the kernel's stat_phase,
    fin_phase and leader): the model runs clean with that, and without it a
    transfer lands in the wrong phase.  (Two shared items, which the host
    never plans, are covered too: the indices are written for any count.)"""
    rng = random.Random(90 + 10 * cluster + shared)
    for _ in range(150):
        occupied = [rng.randint(1, 3276) for _ in range(rng.randint(shared + 1, 9))]
        m = ClusterModel(occupied, cluster, 3, 2, shared=shared)
        status, waits = m.run(rng)
        assert status == "done", (occupied, waits)
        assert m.tail_done == [len(occupied)] * cluster
    with pytest.raises(AssertionError):
        for seed in range(20):
            ClusterModel([3276] * 6, cluster, 3, 2, shared=shared,
                         mistake="uncorrected_phases").run(random.Random(seed))
