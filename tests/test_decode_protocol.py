"""A model of the decode kernel's synchronisation protocol, checked under random schedules.

The latent-attention kernel (one CTA pair per query token and split) coordinates fifteen
warps per CTA and the peer CTA through mbarriers: a TMA thread, the score-MMA and
aggregation-MMA issuers, and three groups of four warps that swap partial scores with
the peer.  Its correctness rests on ordering arguments:
- a parity wait must meet exactly the phase it means;
- a ring slot, score buffer, receive buffer or P buffer is reused only after its last
  reader is done;
- a receive barrier's phase counts the bytes of its own tile only.

This test replays that protocol, role by role and barrier by barrier, as the kernel source
states it. Every warp of both CTAs is an agent. Barriers have mbarrier semantics: arrival
count, transaction bytes that may go transiently negative, and parity waits. Copies,
st.async stores and MMA commits complete at random later times, the commits of one issuing
thread in issue order. Many random schedules run per tile count; a violated argument
shows up as a failed assertion or a deadlock.

With fp8=True it replays the instance for the FP8 cache instead: the TMA thread loads
each tile's E4M3 bytes into staging buffer i % 2 (refilled once tile i-2 was read out of
it); the group that owns the tile (i % 3) widens them into bf16 slot i % 4, tile g before
its first tile and tile i+3 after finishing tile i, after waiting for tile i-2 to be
widened (so the shared staging barrier is in the phase of tile i) and for PV(i-4) to
release the slot; both products read that slot (no second read for PV).

It is a design-level check of the protocol, not of the CUDA code: a change to the
kernel's barriers or buffers must be mirrored here.
"""
import random

import pytest

LAT, ROPE, VBYTES, QROPE, RECV, SIG, LAT8, QLAT = 32768, 4096, 32768, 8192, 16384, 4, 16384, 65536


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
        # mbarrier.try_wait.parity: true once the phase of that parity has completed,
        # i.e. the current (incomplete) phase has the other parity.
        return (self.phase & 1) != parity


class Delay:
    """Not a barrier: a warp that is simply late (scheduled late, or stalled) until `until`."""

    def __init__(self, sim, until):
        self.sim, self.until, self.name, self.phase = sim, until, "delay", None

    def parity_done(self, parity):
        return self.sim.step_no >= self.until


class Slot:
    def __init__(self):
        self.tile = None
        self.landed = False
        self.done = True      # its last reader is finished


class CTA:
    def __init__(self, rank, n):
        self.rank, self.n = rank, n
        B = Bar
        self.qkfull = [B(f"r{rank}.QkFull{i}", 1) for i in range(3)]
        self.ropefull = [B(f"r{rank}.RopeFull{i}", 1) for i in range(2)]
        self.vfull = [B(f"r{rank}.VFull{i}", 1) for i in range(2)]
        self.vempty = [B(f"r{rank}.VEmpty{i}", 1) for i in range(2)]
        self.sfull = [B(f"r{rank}.SFull{g}", 1) for g in range(3)]
        self.sfree = [B(f"r{rank}.SFree{g}", 4) for g in range(3)]
        self.recvfull = [B(f"r{rank}.RecvFull{g}", 1) for g in range(3)]
        self.recvfree = [B(f"r{rank}.RecvFree{b}", 1) for b in range(2)]
        self.freeseen = [B(f"r{rank}.FreeSeen{g}", 4) for g in range(3)]
        self.sigsent = [B(f"r{rank}.SigSent{g}", 4) for g in range(3)]
        self.mref = [B(f"r{rank}.Mref{g}", 128) for g in range(3)]
        self.pvdone = [B(f"r{rank}.PvDone{g}", 1) for g in range(3)]
        self.pfull = B(f"r{rank}.PFull", 128)
        self.qfull = B(f"r{rank}.QFull", 1)
        self.qready = B(f"r{rank}.QReady", 256)
        self.vgo = B(f"r{rank}.VGo", 1)
        # Buffers: which tile occupies them, and whether its readers are done.
        self.qk_slot = [Slot() for _ in range(3)]
        self.rope_slot = [Slot() for _ in range(2)]
        self.v_slot = [Slot() for _ in range(2)]
        # bf16 cache: q~ is staged in the V ring; groups 0 and 1 (eight warps) read it.
        self.q_lat = {"landed": False, "read": [False] * 8}
        self.s_buf = [{"tile": None, "read": [True] * 4} for _ in range(2)]
        self.recv = [{"tile": None, "landed": [False] * 4, "read": [True] * 4} for _ in range(2)]
        self.p_buf = {"tile": None, "written": [False] * 4, "consumed": True}
        self.mref_tile = [None] * 4          # per lane quarter: which tile wrote the reference
        # FP8 instance: staging buffers (one per group) and widened bf16 slots.
        self.stageloaded = [B(f"r{rank}.StageLoaded{i}", 1) for i in range(2)]
        self.stagefree = [B(f"r{rank}.StageFree{i}", 4) for i in range(2)]
        self.slotfull = [B(f"r{rank}.SlotFull{i}", 128) for i in range(4)]
        self.slotempty = [B(f"r{rank}.SlotEmpty{i}", 1) for i in range(4)]
        self.stage = [{"tile": None, "landed": False, "read": [True] * 4} for _ in range(2)]
        self.slot8 = [{"tile": None, "written": [False] * 4, "done": True} for _ in range(4)]
        # The first waits on the "free" barriers are for tiles 2 and 3 (one thread at set-up).
        if n > 2:
            self.recvfree[0].arrive(1, tx=4 * SIG)
        if n > 3:
            self.recvfree[1].arrive(1, tx=4 * SIG)


class Sim:
    def __init__(self, n, seed, partial_last, faults=(), fp8=False):
        self.n = n
        self.fp8 = fp8
        self.faults = set(faults)   # rules left out, to show that the checks catch them
        self.rng = random.Random(seed)
        self.partial_last = partial_last
        self.cta = [CTA(0, n), CTA(1, n)]
        self.agents = []
        self.events = []        # (ready_step, fn) unordered completions (TMA, st.async)
        self.queues = {}        # issuing thread -> list of (ready_step, fn), completed in order
        self.step_no = 0
        for r in range(2):
            c = self.cta[r]
            self.agents.append(self.tma(c))
            self.agents.append(self.qk(c))
            self.agents.append(self.pv(c))
            for g in range(3):
                for q in range(4):
                    self.agents.append(self.group_warp(c, self.cta[1 - r], g, q))

    # ---- asynchronous completions
    def later(self, fn):
        # Copies and remote stores usually land soon, now and then very late: the
        # protocol may not depend on how long any of them takes.
        delay = self.rng.randint(1, 40) if self.rng.random() < 0.95 else self.rng.randint(200, 3000)
        self.events.append((self.step_no + delay, fn))

    def later_in_order(self, queue, fn):
        q = self.queues.setdefault(queue, [])
        ready = max([self.step_no] + [t for t, _ in q]) + self.rng.randint(1, 20)
        q.append((ready, fn))

    # ---- roles (each yields ("wait", bar, phase_index) or None to let others run)
    def tma(self, c):
        n = self.n
        q_issued = False

        def load_q():
            if self.fp8:
                c.qfull.arrive(1, tx=QROPE)
                self.later(lambda: c.qfull.complete_tx(QROPE))
                return
            c.qfull.arrive(1, tx=QROPE + QLAT)

            def land():
                c.q_lat["landed"] = True
                c.qfull.complete_tx(QROPE + QLAT)
            self.later(land)

        for i in range(n):
            if i >= 1 and not q_issued:
                load_q()
                q_issued = True
            if self.fp8:
                if i >= 2 and "no_stagefree" not in self.faults:
                    yield ("wait", c.stagefree[i % 2], i // 2 - 1)
                st = c.stage[i % 2]
                check(all(st["read"]), f"r{c.rank}: staging {i % 2} refilled for tile {i} before tile {st['tile']} was read")
                st["tile"], st["landed"], st["read"] = i, False, [False] * 4
                c.stageloaded[i % 2].arrive(1, tx=LAT8)

                def land8(st=st, i=i):
                    st["landed"] = True
                    c.stageloaded[i % 2].complete_tx(LAT8)
                self.later(land8)
                yield None
            if self.fp8:
                pass
            elif i == 3 and "no_vgo" not in self.faults:
                yield ("wait", c.vgo, 0)
            if not self.fp8:
                if i >= 3:
                    yield ("wait", c.sfull[(i - 3) % 3], (i - 3) // 3)
                s = c.qk_slot[i % 3]
                check(s.done, f"r{c.rank}: latent slot {i % 3} refilled for tile {i} before QK of tile {s.tile} finished")
                s.tile, s.landed, s.done = i, False, False
                c.qkfull[i % 3].arrive(1, tx=LAT)

                def land_lat(s=s, i=i):
                    s.landed = True
                    c.qkfull[i % 3].complete_tx(LAT)
                self.later(land_lat)
                yield None
            if i >= 2:
                yield ("wait", c.sfull[(i - 2) % 3], (i - 2) // 3)
            rs = c.rope_slot[i % 2]
            check(rs.done, f"r{c.rank}: rope slot {i % 2} refilled for tile {i} before QK of tile {rs.tile} finished")
            rs.tile, rs.landed, rs.done = i, False, False
            c.ropefull[i % 2].arrive(1, tx=ROPE)

            def land_rope(rs=rs, i=i):
                rs.landed = True
                c.ropefull[i % 2].complete_tx(ROPE)
            self.later(land_rope)
            yield None
        if not q_issued:
            load_q()

    def qk(self, c):
        n = self.n
        yield ("wait", c.qfull, 0)
        yield ("wait", c.qready, 0)
        for i in range(n):
            if i >= 2 and "no_sfree" not in self.faults:
                yield ("wait", c.sfree[(i - 2) % 3], (i - 2) // 3)
            sb = c.s_buf[i & 1]
            if self.fp8:
                yield ("wait", c.slotfull[i % 4], i // 4)
                s8 = c.slot8[i % 4]
                check(s8["tile"] == i and all(s8["written"]), f"r{c.rank}: QK({i}) reads a slot not holding tile {i}")
                s = Slot()
            else:
                yield ("wait", c.qkfull[i % 3], i // 3)
                s = c.qk_slot[i % 3]
                check(s.tile == i and s.landed, f"r{c.rank}: QK({i}) reads a latent slot that does not hold tile {i}")
            check(all(sb["read"]), f"r{c.rank}: QK({i}) overwrites S buffer {i & 1} before tile {sb['tile']} was read")
            sb["tile"], sb["read"] = i, [False] * 4
            yield ("wait", c.ropefull[i % 2], i // 2)
            rs = c.rope_slot[i % 2]
            check(rs.tile == i and rs.landed, f"r{c.rank}: QK({i}) reads a rope slot that does not hold tile {i}")

            def done(i=i, s=s, rs=rs):
                s.done = True
                rs.done = True
                c.sfull[i % 3].arrive()
            self.later_in_order(("qk", c.rank), done)
            yield None

    def pv(self, c):
        n = self.n

        def load_v(i):
            v = c.v_slot[i % 2]
            check(v.done, f"r{c.rank}: V slot {i % 2} refilled for tile {i} before PV of tile {v.tile} finished")
            check(all(c.q_lat["read"]), f"r{c.rank}: V slot {i % 2} refilled for tile {i} while q~ is still unread")
            v.tile, v.landed, v.done = i, False, False
            c.vfull[i % 2].arrive(1, tx=VBYTES)

            def land(v=v):
                v.landed = True
                c.vfull[i % 2].complete_tx(VBYTES)
            self.later(land)

        if self.rng.random() < 0.3:     # the issuer may start late
            yield ("wait", Delay(self, self.step_no + self.rng.randint(1, 400)), 0)
        if self.fp8:
            for i in range(n):
                yield ("wait", c.pfull, i)
                p, s8 = c.p_buf, c.slot8[i % 4]
                check(p["tile"] == i and all(p["written"]), f"r{c.rank}: PV({i}) reads a P buffer not holding tile {i}")
                check(s8["tile"] == i and all(s8["written"]), f"r{c.rank}: PV({i}) reads a slot not holding tile {i}")

                def done8(i=i, s8=s8, p=p):
                    s8["done"] = True
                    p["consumed"] = True
                    c.slotempty[i % 4].arrive()
                    c.pvdone[i % 3].arrive()
                self.later_in_order(("pv", c.rank), done8)
                yield None
            return
        if "no_qready_v" not in self.faults:
            yield ("wait", c.qready, 0)      # the V ring holds q~ until it is in TMEM
        for i in range(min(2, n)):
            # The first V tiles are requested once the same rows have landed in the score
            # ring (phase 0 of its slot), so that they come from L2.
            yield ("wait", c.qkfull[i], 0)
            s = c.qk_slot[i]
            check(s.tile == i and s.landed, f"r{c.rank}: first V({i}) follows a slot that no longer holds tile {i}")
            load_v(i)
        c.vgo.arrive()
        for i in range(n):
            vs = i % 2
            if i + 1 < n and i + 1 >= 2:
                yield ("wait", c.vempty[(i + 1) % 2], (i + 1) // 2 - 1)
                load_v(i + 1)
            yield ("wait", c.pfull, i)
            yield ("wait", c.vfull[vs], i // 2)
            p, v = c.p_buf, c.v_slot[vs]
            check(p["tile"] == i and all(p["written"]), f"r{c.rank}: PV({i}) reads a P buffer that does not hold tile {i}")
            check(v.tile == i and v.landed, f"r{c.rank}: PV({i}) reads a V slot that does not hold tile {i}")

            def done(i=i, v=v, p=p):
                v.done = True
                p["consumed"] = True
                c.vempty[i % 2].arrive()
                c.pvdone[i % 3].arrive()
            self.later_in_order(("pv", c.rank), done)
            yield None

    def convert(self, c, j, q):
        """FP8: this warp's share of widening tile j (staging j % 2 -> slot j % 4)."""
        if j >= 2 and "no_prevwiden" not in self.faults:
            yield ("wait", c.slotfull[(j - 2) % 4], (j - 2) // 4)
        yield ("wait", c.stageloaded[j % 2], j // 2)
        if j >= 4 and "no_slotempty" not in self.faults:
            yield ("wait", c.slotempty[j % 4], j // 4 - 1)
        st, s8 = c.stage[j % 2], c.slot8[j % 4]
        check(st["tile"] == j and st["landed"], f"r{c.rank}: widening tile {j} from staging holding {st['tile']}")
        st["read"][q] = True
        c.stagefree[j % 2].arrive(1)
        if s8["tile"] != j:
            check(s8["done"], f"r{c.rank}: tile {j} overwrites slot {j % 4} before PV of tile {s8['tile']}")
            s8["tile"], s8["written"], s8["done"] = j, [False] * 4, False
        s8["written"][q] = True
        c.slotfull[j % 4].arrive(32)
        yield None

    def group_warp(self, c, peer, g, q):
        n = self.n
        if g < 2:
            if self.fp8:
                c.qready.arrive(32)        # this warp's q~ columns are in TMEM (read from q_cat)
            else:
                yield ("wait", c.qfull, 0)
                check(c.q_lat["landed"], f"r{c.rank} g{g}: q~ read from the V ring before it landed")
                c.q_lat["read"][4 * g + q] = True
                c.qready.arrive(32)        # this warp's q~ columns are in TMEM
        if q == 0 and g < n:
            c.recvfull[g].arrive(1, tx=RECV)
        if self.fp8 and g < n:
            yield from self.convert(c, g, q)
        for i in range(g, n, 3):
            k = i // 3
            b = i & 1
            yield ("wait", c.sfull[g], k)
            sb = c.s_buf[b]
            check(sb["tile"] == i, f"r{c.rank} g{g}: S buffer {b} does not hold tile {i}")
            sb["read"][q] = True
            c.sfree[g].arrive(1)
            yield None
            if i >= 1 and "no_freeseen" not in self.faults:
                yield ("wait", c.freeseen[(i - 1) % 3], (i - 1) // 3)
            if i >= 2:
                yield ("wait", c.recvfree[b], (i - 2) // 2)
                if q == 0 and i + 2 < n:
                    c.recvfree[b].arrive(1, tx=4 * SIG)
            c.freeseen[g].arrive(1)
            # This warp's quarter of the partial scores into the peer's receive buffer b.
            rb = peer.recv[b]
            if rb["tile"] != i:
                check(rb["tile"] is None or (rb["tile"] == i - 2 and all(rb["read"])),
                      f"r{c.rank} g{g}: tile {i} overwrites the peer's buffer {b} before it read tile {rb['tile']}")
                rb["tile"], rb["landed"], rb["read"] = i, [False] * 4, [False] * 4

            def land(rb=rb, g=g):
                rb["landed"][q] = True
                peer.recvfull[g].complete_tx(RECV // 4)
            self.later(land)
            yield None
            yield ("wait", c.recvfull[g], k)
            if q == 0 and i + 3 < n:
                c.recvfull[g].arrive(1, tx=RECV)
            mine = c.recv[b]
            check(mine["tile"] == i and all(mine["landed"]),
                  f"r{c.rank} g{g}: receive phase of tile {i} completed without all of its bytes")
            mine["read"][q] = True
            if i >= 1 and "no_sigsent" not in self.faults:
                yield ("wait", c.sigsent[(i - 1) % 3], (i - 1) // 3)
            if i + 2 < n:
                self.later(lambda b=b: peer.recvfree[b].complete_tx(SIG))
            c.sigsent[g].arrive(1)
            yield None
            if i >= 1:
                yield ("wait", c.mref[(i - 1) % 3], (i - 1) // 3)
                check(c.mref_tile[q] == i - 1, f"r{c.rank} g{g}: reference maximum not from tile {i - 1}")
            c.mref_tile[q] = i
            c.mref[g].arrive(32)
            if i >= 1:
                yield ("wait", c.pvdone[(i - 1) % 3], (i - 1) // 3)
            p = c.p_buf
            if p["tile"] != i:
                check(p["consumed"], f"r{c.rank} g{g}: P of tile {i} overwrites tile {p['tile']} before its PV")
                p["tile"], p["written"], p["consumed"] = i, [False] * 4, False
            p["written"][q] = True
            if i == n - 1 and self.partial_last and not self.fp8:
                yield ("wait", c.vfull[i % 2], i // 2)
                v = c.v_slot[i % 2]
                check(v.tile == i and v.landed, f"r{c.rank} g{g}: clears a V slot that does not hold tile {i}")
            c.pfull.arrive(32)
            yield None
            if self.fp8 and i + 3 < n:
                yield from self.convert(c, i + 3, q)
        yield ("wait", c.pvdone[(n - 1) % 3], (n - 1) // 3)

    # ---- scheduler
    def run(self):
        states = [[a, None] for a in self.agents]     # [generator, pending wait or None]
        live = len(states)
        while live or self.events or any(self.queues.values()):
            self.step_no += 1
            choices = []
            for idx, (gen, wait) in enumerate(states):
                if gen is None:
                    continue
                if wait is None or wait[0].parity_done(wait[1] & 1):
                    choices.append(("agent", idx))
            ready_ev = [j for j, (t, _) in enumerate(self.events) if t <= self.step_no]
            choices += [("event", j) for j in ready_ev]
            for key, q in self.queues.items():
                if q and q[0][0] <= self.step_no:
                    choices.append(("queue", key))
            if not choices:
                delayed = any(w is not None and isinstance(w[0], Delay) for g, w in states if g is not None)
                if self.events or any(self.queues.values()) or delayed:
                    continue                     # only time passes
                stuck = [w for g, w in states if g is not None]
                raise ProtocolError(f"deadlock: waits {[(w[0].name, w[1]) for w in stuck if w]}")
            kind, which = self.rng.choice(choices)
            if kind == "event":
                _, fn = self.events.pop(which)
                fn()
            elif kind == "queue":
                _, fn = self.queues[which].pop(0)
                fn()
            else:
                gen, wait = states[which]
                if wait is not None and not isinstance(wait[0], Delay):
                    bar, k = wait
                    check(bar.phase == k + 1,
                          f"{bar.name}: a wait for phase {k} returned with {bar.phase} phases complete")
                try:
                    act = next(gen)
                except StopIteration:
                    states[which] = [None, None]
                    live -= 1
                    continue
                states[which][1] = (act[1], act[2]) if act else None
        return True


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8, 13])
@pytest.mark.parametrize("partial_last", [False, True])
def test_protocol_holds_under_random_schedules(n, partial_last):
    for seed in range(40):
        assert Sim(n, seed, partial_last).run()


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8, 13])
def test_fp8_protocol_holds_under_random_schedules(n):
    for seed in range(40):
        assert Sim(n, seed, seed % 2 == 1, fp8=True).run()


@pytest.mark.parametrize("fault", ["no_prevwiden", "no_stagefree"])
def test_the_fp8_model_catches_a_broken_rule(fault):
    # - no_prevwiden: the group waits for tile i's bytes in the shared staging buffer
    #   without first waiting for tile i-2 to be widened, so its parity wait can take the
    #   phase of tile i-2 (the mistake of an earlier version of this instance);
    # - no_stagefree: tile i is loaded into staging buffer i % 2 before tile i-2 was read.
    # Some schedule must trip an assertion or deadlock.
    failures = 0
    for seed in range(200):
        for n in (7, 13):
            try:
                Sim(n, seed, False, faults=[fault], fp8=True).run()
            except ProtocolError:
                failures += 1
    assert failures > 0, f"no schedule exposed {fault}"


@pytest.mark.parametrize("n", [5, 7, 13])
def test_fp8_slot_empty_wait_is_implied(n):
    # The group also waits for PV(i-4) before widening tile i into slot i % 4 (kSlotEmpty).
    # The model shows it is implied: the group widens tile i after finishing tile i-3, for
    # which it waited for PV(i-4).  Without it every schedule holds.
    for seed in range(60):
        assert Sim(n, seed, False, faults=["no_slotempty"], fp8=True).run()


@pytest.mark.parametrize("fault", ["no_sfree", "no_freeseen", "no_vgo", "no_qready_v"])
def test_the_model_catches_a_broken_rule(fault):
    # Each planted mistake leaves out one rule of the protocol:
    # - no_qready_v: the aggregation issuer requests the first V tiles before groups 0 and
    #   1 have moved q~ out of the V ring;
    # - no_sfree: the score issuer overwrites S buffer i & 1 before the group of tile i-2
    #   read it;
    # - no_freeseen: the groups wait for the peer's "free" signals out of tile order, so a
    #   parity wait can meet the phase of another tile;
    # - no_vgo: tile 3 is requested before the aggregation issuer has seen tile 0 land,
    #   so its phase-0 wait on that slot can meet a later phase.
    # Some schedule must then trip an assertion or deadlock.
    failures = 0
    for seed in range(200):
        for n in (7, 13):
            try:
                Sim(n, seed, False, faults=[fault]).run()
            except ProtocolError:
                failures += 1
    assert failures > 0, f"no schedule exposed {fault}"


@pytest.mark.parametrize("n", [4, 7, 13])
def test_signal_order_chain_is_implied(n):
    # The kernel also sends its "free" signals in tile order (kSigSent), so that the
    # peer's tile i+3 cannot land on a group's receive barrier before that group's phase
    # of tile i completed.  The model shows the rule is already implied: the peer sends
    # tile i+3 only after passing, in tile order (kFreeSeen), its wait for tile i+2, which
    # needs our signal for tile i, which follows our read of tile i.  Without the chain,
    # every schedule still holds.
    for seed in range(60):
        for partial_last in (False, True):
            assert Sim(n, seed, partial_last, faults=["no_sigsent"]).run()
