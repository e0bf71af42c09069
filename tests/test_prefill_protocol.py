"""A model of the persistent prefill attention kernel's synchronisation, checked under
random schedules.

Each CTA of the prefill kernel walks a list of work items (sequence, head, 128 queries)
and keeps its rings running from one item to the next. Four agents share these buffers
through mbarriers: a key-tile TMA thread (which also loads each item's q^R), a value-tile
TMA thread (which also stores each item's O), the MMA thread, and the softmax warps. The
softmax warps are modelled as one agent, since they meet at named barriers for every tile.
The buffers are:
- the key ring (2 stages) and the value ring (2 stages);
- q^R and two 16 KB slots in shared memory;
- q_nope, the two score buffers and O in TMEM. P(g) is written into the score buffer of
  S(g), so P is double-buffered with S.

The slots carry the next item's q_nope in (loaded by the softmax leader a tile before an
item's last) and half of an item's O out. The other half goes out through the value stage
of the item's last tile. The value thread stores O before it loads that stage again.

Each buffer is reused only after its last reader is done. The checks are:
- the key stage of tile g is reloaded only after the score products of g-2;
- q^R and q_nope of item n+1 are written only after the last score products of item n;
- the first aggregation of item n+1 (which overwrites O) starts only after the softmax
  warps have read out O of item n (implied: they write its P after that);
- S(g) overwrites P(g-2) only after PV(g-2) has been issued (the MMAs of one thread run
  in issue order, so PV(g-2) has read P(g-2) by then);
- O is rescaled (at a tile where a row's maximum grows) only after PV(g-1), and read out
  only after the item's last PV;
- the slots take q_nope only after the previous O has been read out of them, and O only
  after that q_nope has been moved to TMEM;
- a value stage takes O only after its PV, and the next tile only after O has been read
  out of it;
- and so on for the score buffers and the value ring.

Copies complete at random later times. MMA commits complete in issue order, also later.
A wait returns only on the phase it means (parity semantics, with the phase checked):
the softmax waits for the PV barriers only now and then, so this also checks that such a
barrier is never two phases past the one waited for.
A rule left out shows up as a failed check or a deadlock.

The item list restates the kernel's schedule: unit u (dealt round-robin over the CTAs) is
(sequence, head) u // npu with query blocks n_qb-1-i and i (i = u % npu).

It is a design-level check of the protocol, not of the CUDA code: a change to the kernel's
barriers or buffers must be mirrored here.
"""
import random

import pytest


class ProtocolError(AssertionError):
    pass


def check(cond, msg):
    if not cond:
        raise ProtocolError(msg)


class Bar:
    """An mbarrier: `count` arrivals plus a zero transaction count complete a phase."""

    def __init__(self, name, count):
        self.name, self.count = name, count
        self.pending, self.tx, self.phase = count, 0, 0

    def arrive(self, n=1, tx=0):
        self.tx += tx
        self.pending -= n
        check(self.pending >= 0, f"{self.name}: more arrivals than its count in one phase")
        self._maybe_complete()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._maybe_complete()

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def parity_done(self, parity):
        return (self.phase & 1) != parity


def items_of_cta(c, grid, B, H, T_q, T_kv):
    n_qb = (T_q + 127) // 128
    npu = (n_qb + 1) // 2
    units = B * H * npu
    out = []
    for u in range(c, units, grid):
        i = u % npu
        for qb in ([n_qb - 1 - i] + ([i] if i < n_qb - 1 - i else [])):
            q0 = qb * 128
            last = min(T_kv - 1, T_kv - T_q + min(q0 + 127, T_q - 1))
            out.append(last // 128 + 1)          # key tiles of the item
    return out


KT, VT, QR = 3 * 16384, 2 * 16384, 16384


class Sim:
    def __init__(self, nts, seed, faults=()):
        self.nts = nts                         # key tiles of each item of this CTA
        self.faults = set(faults)
        self.rng = random.Random(seed)
        B = Bar
        self.qfull, self.qready = B("QFull", 1), B("QReady", 256)
        self.qrfree = B("QrFree", 1)
        self.kfull = [B(f"KFull{i}", 1) for i in range(2)]
        self.kempty = [B(f"KEmpty{i}", 1) for i in range(2)]
        self.vfull = [B(f"VFull{i}", 1) for i in range(2)]
        self.vempty = [B(f"VEmpty{i}", 1) for i in range(2)]
        self.sfull = [B(f"SFull{i}", 1) for i in range(2)]
        self.sfree = [B(f"SFree{i}", 8) for i in range(2)]
        self.pfull = [B(f"PFull{i}", 256) for i in range(2)]
        if "one_pfull" in self.faults:      # one P barrier for all tiles: phase g, not g // 2
            self.pfull = [self.pfull[0]] * 2
        self.pf = (lambda t: (self.pfull[0], t)) if "one_pfull" in self.faults else \
            (lambda t: (self.pfull[t & 1], t // 2))
        self.pvdone = [B(f"PvDone{i}", 1) for i in range(2)]
        self.qnfull, self.ostaged, self.oread = B("QnFull", 1), B("OStaged", 256), B("ORead", 1)
        # Buffer state: occupant and whether its readers are done.
        self.kslot = [{"tile": None, "landed": False, "done": True} for _ in range(2)]
        self.vslot = [{"tile": None, "landed": False, "done": True, "o": None} for _ in range(2)]
        self.slots = {"what": None, "landed": True, "read": True}   # ("q", n) or ("o", n)
        self.qrope = {"item": None, "landed": False, "done": True}
        self.qnope = {"item": None, "done": True}
        self.sbuf = [{"tile": None, "ready": False, "read": True, "p": None, "p_issued": True}
                     for _ in range(2)]
        self.o = {"item": None, "pvs": 0, "read": True}
        self.qk_done = {}                       # tile -> score products complete
        self.item_of = []                       # tile -> item
        self.first = []                         # tile -> first tile of its item
        self.last = []
        for n, nt in enumerate(nts):
            for j in range(nt):
                self.item_of.append(n)
                self.first.append(j == 0)
                self.last.append(j == nt - 1)
        self.events, self.mma_queue, self.step_no = [], [], 0
        self.agents = [self.kprod(), self.vprod(), self.mma(), self.softmax()]

    def later(self, fn):
        delay = self.rng.randint(1, 40) if self.rng.random() < 0.95 else self.rng.randint(200, 2000)
        self.events.append((self.step_no + delay, fn))

    def commit(self, fn):   # tcgen05.commit: completes after every earlier MMA, in order
        ready = max([self.step_no] + [t for t, _ in self.mma_queue]) + self.rng.randint(1, 30)
        self.mma_queue.append((ready, fn))

    # ---- the key-tile producer (and q^R)
    def kprod(self):
        g = 0
        for n, nt in enumerate(self.nts):
            for j in range(nt):
                ks = g % 2
                if g >= 2 and "no_kempty" not in self.faults:
                    yield ("wait", self.kempty[ks], g // 2 - 1)
                s = self.kslot[ks]
                check(s["done"], f"key stage {ks} reloaded for tile {g} before S({s['tile']}) was done")
                s.update(tile=g, landed=False, done=False)
                self.kfull[ks].arrive(1, tx=KT)

                def land(s=s, ks=ks):
                    s["landed"] = True
                    self.kfull[ks].complete_tx(KT)
                self.later(land)
                if j == 0:
                    if n > 0 and "no_qrfree" not in self.faults:
                        yield ("wait", self.qrfree, n - 1)
                    check(self.qrope["done"], f"q^R of item {n} loaded before the score products of item "
                                              f"{self.qrope['item']} were done")
                    self.qrope.update(item=n, landed=False, done=False)
                    self.qfull.arrive(1, tx=QR)

                    def landq():
                        self.qrope["landed"] = True
                        self.qfull.complete_tx(QR)
                    self.later(landq)
                g += 1
                yield None

    # ---- the value-tile producer, which also stores O
    def store_o(self, n, last):
        if "no_ostaged" not in self.faults:
            yield ("wait", self.ostaged, n)
        vs = self.vslot[last % 2]
        check(self.slots["what"] == ("o", n) and vs["o"] == n, f"O of item {n} stored from slots holding "
                                                               f"{self.slots['what']} and a stage holding {vs['o']}")
        done = Bar("StoreRead", 1)

        def read():
            self.slots["read"] = True
            vs["o"] = None
            done.arrive()
        self.later(read)
        yield ("wait", done, 0)
        self.oread.arrive()

    def vprod(self):
        g = 0
        pend = []
        for n, nt in enumerate(self.nts):
            for j in range(nt):
                vs = g % 2
                if g >= 2:
                    yield ("wait", self.vempty[vs], g // 2 - 1)
                if pend and pend[0][1] + 2 == g:
                    yield from self.store_o(*pend.pop(0))
                s = self.vslot[vs]
                check(s["done"] and s["o"] is None, f"value stage {vs} reloaded for tile {g} before PV({s['tile']}) "
                                                    f"was done or while it holds O of item {s['o']}")
                s.update(tile=g, landed=False, done=False)
                self.vfull[vs].arrive(1, tx=VT)

                def land(s=s, vs=vs):
                    s["landed"] = True
                    self.vfull[vs].complete_tx(VT)
                self.later(land)
                g += 1
                yield None
            pend.append((n, g - 1))
        while pend:
            yield from self.store_o(*pend.pop(0))

    # ---- the MMA issuer
    def pv(self, gi):
        n = self.item_of[gi]
        yield ("wait", *self.pf(gi))
        yield ("wait", self.vfull[gi % 2], gi // 2)
        sb = self.sbuf[gi & 1]
        check(sb["p"] == gi and not sb["p_issued"], f"PV({gi}) read P of tile {sb['p']}")
        sb["p_issued"] = True        # read before any later MMA of this thread writes the buffer
        vs = self.vslot[gi % 2]
        check(vs["tile"] == gi and vs["landed"], f"PV({gi}) read value stage holding {vs['tile']}")
        if self.first[gi]:
            check(self.o["read"], f"PV({gi}) overwrote O of item {self.o['item']} before it was read out")
            self.o.update(item=n, pvs=0, read=False)
        else:
            check(self.o["item"] == n, f"PV({gi}) added into O of item {self.o['item']}")

        def done():
            vs["done"] = True
            self.vempty[gi % 2].arrive()
            self.o["pvs"] += 1
            self.pvdone[gi & 1].arrive()
        self.commit(done)

    def mma(self):
        pend = None
        g = 0
        for n, nt in enumerate(self.nts):
            if pend is not None:
                yield from self.pv(pend)
                pend = None
            yield ("wait", self.qfull, n)
            yield ("wait", self.qready, n)
            for j in range(nt):
                if g >= 2:
                    yield ("wait", self.sfree[g & 1], g // 2 - 1)
                yield ("wait", self.kfull[g % 2], g // 2)
                ks = self.kslot[g % 2]
                check(ks["tile"] == g and ks["landed"], f"S({g}) read key stage holding {ks['tile']}")
                check(self.qrope["item"] == n and self.qrope["landed"], f"S({g}) read q^R of item {self.qrope['item']}")
                check(self.qnope["item"] == n, f"S({g}) read q_nope of item {self.qnope['item']}")
                sb = self.sbuf[g & 1]
                check(sb["read"], f"S({g}) overwrote S({sb['tile']}) before the softmax read it")
                check(sb["p"] is None or sb["p_issued"], f"S({g}) overwrote P({sb['p']}) before its PV was issued")
                sb.update(tile=g, ready=False, read=False, p=None, p_issued=True)

                def sdone(g=g, sb=sb, ks=ks, last=(j == nt - 1), n=n):
                    sb["ready"] = True
                    self.sfull[g & 1].arrive()
                    ks["done"] = True
                    self.kempty[g % 2].arrive()
                    if last:
                        self.qrope["done"] = True
                        self.qnope["done"] = True
                        self.qrfree.arrive()
                self.commit(sdone)
                if pend is not None:
                    yield from self.pv(pend)
                pend = g
                g += 1
                yield None
        if pend is not None:
            yield from self.pv(pend)

    # ---- the softmax warps
    def softmax(self):
        def q_issue(n):   # the leader loads q_nope of item n into the slots
            check(self.slots["read"], f"q_nope of item {n} loaded into slots holding unread {self.slots['what']}")
            self.slots.update(what=("q", n), landed=False, read=False)
            self.qnfull.arrive(1, tx=2 * QR)

            def land():
                self.slots["landed"] = True
                self.qnfull.complete_tx(2 * QR)
            self.later(land)

        def q_move(n):    # every thread moves its half row into TMEM
            yield ("wait", self.qnfull, n)
            check(self.slots["what"] == ("q", n) and self.slots["landed"], f"q_nope of item {n} read from slots "
                                                                           f"holding {self.slots['what']}")
            check(self.qnope["done"], f"q_nope of item {n} written while item {self.qnope['item']} still reads it")
            self.slots["read"] = True
            self.qnope.update(item=n, done=False)
            self.qready.arrive(256)

        g = 0
        nitems = len(self.nts)
        q_issue(0)
        yield from q_move(0)
        for n, nt in enumerate(self.nts):
            j_q = max(0, nt - 2)
            for j in range(nt):
                if n + 1 < nitems and j == j_q:
                    if n > 0 and "no_oread" not in self.faults:
                        yield ("wait", self.oread, n - 1)
                    q_issue(n + 1)
                if j == nt - 1 and n + 1 < nitems and "early_qmove" in self.faults:
                    yield from q_move(n + 1)
                yield ("wait", self.sfull[g & 1], g // 2)
                sb = self.sbuf[g & 1]
                check(sb["tile"] == g and sb["ready"], f"softmax of tile {g} read S({sb['tile']})")
                sb["read"] = True
                self.sfree[g & 1].arrive(8)
                if j > 0 and self.rng.random() < 0.3:   # a row's maximum grew: O is rescaled
                    if "no_pvdone" not in self.faults:
                        yield ("wait", self.pvdone[(g - 1) & 1], (g - 1) // 2)
                    check(self.o["item"] == n and self.o["pvs"] == j,
                          f"O rescaled at tile {g} with {self.o['pvs']} of its item's {j} earlier PVs done")
                check(sb["p"] is None, f"P({g}) written over P({sb['p']})")
                sb.update(p=g, p_issued=False)
                if self.rng.random() < 0.3:      # a partial tile: rows past the end cleared
                    yield ("wait", self.vfull[g % 2], g // 2)
                    check(self.vslot[g % 2]["tile"] == g, f"cleared the value stage of tile {self.vslot[g % 2]['tile']}")
                self.pf(g)[0].arrive(256)
                if j == nt - 1 and n + 1 < nitems and "early_qmove" not in self.faults:
                    yield from q_move(n + 1)
                g += 1
                yield None
            if "no_pvdone_epi" not in self.faults:
                yield ("wait", self.pvdone[(g - 1) & 1], (g - 1) // 2)
            check(self.o["item"] == n and self.o["pvs"] == nt, f"O of item {n} read out with {self.o['pvs']} of {nt} PVs")
            self.o["read"] = True
            if n + 1 == nitems and n > 0:
                yield ("wait", self.oread, n - 1)
            check(self.slots["read"], f"O of item {n} staged into slots holding unread {self.slots['what']}")
            vs = self.vslot[(g - 1) % 2]
            check(vs["tile"] == g - 1 and vs["done"] and vs["o"] is None,
                  f"O of item {n} staged into the value stage of tile {vs['tile']} (PV done: {vs['done']})")
            self.slots.update(what=("o", n), landed=True, read=False)
            vs["o"] = n
            self.ostaged.arrive(256)
            yield None

    def run(self):
        states = [[a, None] for a in self.agents]
        live = len(states)
        while live or self.events or self.mma_queue:
            self.step_no += 1
            choices = [("agent", i) for i, (gen, w) in enumerate(states)
                       if gen is not None and (w is None or w[0].parity_done(w[1] & 1))]
            choices += [("event", j) for j, (t, _) in enumerate(self.events) if t <= self.step_no]
            if self.mma_queue and self.mma_queue[0][0] <= self.step_no:
                choices.append(("mma", 0))
            if not choices:
                if self.events or self.mma_queue:
                    continue
                raise ProtocolError(f"deadlock: waits {[(w[0].name, w[1]) for g_, w in states if g_ and w]}")
            kind, which = self.rng.choice(choices)
            if kind == "event":
                self.events.pop(which)[1]()
            elif kind == "mma":
                self.mma_queue.pop(0)[1]()
            else:
                gen, w = states[which]
                if w is not None:
                    check(w[0].phase == w[1] + 1, f"{w[0].name}: a wait for phase {w[1]} returned with "
                                                  f"{w[0].phase} phases complete")
                try:
                    act = next(gen)
                except StopIteration:
                    states[which] = [None, None]
                    live -= 1
                    continue
                states[which][1] = (act[1], act[2]) if act else None
        return True


# (B, H, T_q, T_kv): the prompt and chunk shapes of the GPU tests; the CTAs checked are
# the first few and the last, with grids of 148 SMs.
SHAPES = [(1, 128, 4096, 4096), (2, 16, 300, 300), (1, 16, 130, 700), (1, 128, 200, 1000),
          (2, 64, 600, 900), (1, 128, 1024, 1024)]


def test_schedule_covers_every_item_once():
    for B, H, T_q, T_kv in SHAPES:
        n_qb = (T_q + 127) // 128
        npu = (n_qb + 1) // 2
        grid = min(B * H * npu, 148)
        total = sum(len(items_of_cta(c, grid, B, H, T_q, T_kv)) for c in range(grid))
        assert total == B * H * n_qb


@pytest.mark.parametrize("shape", SHAPES)
def test_protocol_holds_under_random_schedules(shape):
    B, H, T_q, T_kv = shape
    n_qb = (T_q + 127) // 128
    grid = min(B * H * ((n_qb + 1) // 2), 148)
    for c in sorted({0, 1, grid - 1}):
        nts = items_of_cta(c, grid, B, H, T_q, T_kv)
        for seed in range(6 if len(nts) > 8 else 30):
            assert Sim(nts, seed).run()


@pytest.mark.parametrize("fault", ["no_qrfree", "no_kempty", "no_pvdone", "no_pvdone_epi", "one_pfull",
                                   "early_qmove", "no_ostaged", "no_oread"])
def test_the_model_catches_a_broken_rule(fault):
    # - no_qrfree: q^R of the next item is loaded without waiting for the last score
    #   products of the current one;
    # - no_kempty: a key stage is reloaded without waiting for the score products of the
    #   tile two back;
    # - no_pvdone: O is rescaled without waiting for PV(g-1);
    # - no_pvdone_epi: O is read out without waiting for the item's last PV;
    # - one_pfull: one P barrier for every tile, which the softmax can move two phases past
    #   the MMA thread's wait;
    # - early_qmove: the next item's q_nope is moved into TMEM before the softmax has seen
    #   the item's last scores (whose products may still read the current q_nope);
    # - no_ostaged: O is stored without waiting for the softmax warps to stage it;
    # - no_oread: the next q_nope is loaded into the slots without waiting for the previous
    #   O to be read out of them.
    caught = 0
    for seed in range(40):
        try:
            Sim([3, 1, 2, 2], seed, faults=[fault]).run()
        except ProtocolError:
            caught += 1
    assert caught > 0
