"""A host-side model of the multi-query kernel's synchronisation protocol
(paged_prefill_tc_kernel in csrc/prefill_tc.cuh), run under random
interleavings.

The kernel's roles meet only through mbarriers whose waits test a phase
*parity*: a wait for phase k passes as soon as the barrier's current phase
has the other parity, so it cannot tell phase k from phase k - 2.  Whether
every wait is at most one phase away depends on the order in which the roles
fill and free the shared-memory ring of K/V sub-tiles, the unit ring, the Q
buffers, the S/P and O regions of TMEM.  This model replays that order with
the same position arithmetic as the kernel (ring positions of K(t) and V(t),
one or two Q buffers and O accumulators by head_dim, NPROD producer warps
taking positions round robin) and checks, for every interleaving it draws:

* no parity wait passes while the phase it waits for is still open;
* a slot is re-armed only after every MMA reading it has finished;
* every MMA reads a slot (or Q buffer) holding the position it expects, landed;
* O is not overwritten during its epilogue, and S(t + 2) does not overwrite
  S(t) before the softmax has read it.

The tensor pipe completes MMAs and commits in issue order; TMA copies land in
any order.  It also shows that the model has teeth: with the claim order of
an earlier version (the previous unit's last PV issued before the new unit's
first S only when the new Q had not landed yet) it finds a stale parity pass.
"""
import random
from collections import deque

import pytest


class StaleWait(AssertionError):
    pass


class Bar:
    """mbarrier: expected arrival count, transaction bytes, completed phases."""

    def __init__(self, name, count):
        self.name, self.count = name, count
        self.pending, self.tx, self.phase = count, 0, 0

    def arrive(self, tx=0):
        self.tx += tx
        self.pending -= 1
        assert self.pending >= 0, f"{self.name}: more arrivals than expected in a phase"
        self._advance()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._advance()

    def _advance(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def try_wait(self, parity):
        return (self.phase & 1) != parity


def units_of(lengths, D, G, prior=None, causal=True):
    """The kernel's work units (request, query block) for one KV head: key
    tiles and keys read, heaviest block first within a request."""
    BQ = 128 // G
    out = []
    for r, n in enumerate(lengths):
        N = n + (prior[r] if prior else 0)
        nblk = (n + BQ - 1) // BQ
        for lp in range(nblk):
            i0 = (nblk - 1 - lp) * BQ
            rows = min(BQ, n - i0)
            kend = max(0, min(N, N - n + i0 + rows)) if causal else N
            out.append({"ntiles": (kend + 127) // 128, "kend": kend})
    return out


def simulate(D, units, nprod, seed, order="fixed"):
    rnd = random.Random(seed)
    SUB = D // 64
    NSLOT = 10 if D >= 128 else 12
    NQB = 1 if D >= 256 else 2
    NOB = 1 if D >= 256 else 2
    NU, BN = 8, 128
    VKEYS = BN // SUB
    PV_FIRST = NQB == 1

    def pos_k(t, unit_first):
        if t == 0:
            return 0
        return (2 * t - 1) * SUB + (SUB if (PV_FIRST and unit_first and order == "fixed") else 0)

    def pos_v(t, unit_last):
        if PV_FIRST and order == "fixed":
            return (2 * t + 1) * SUB + (0 if unit_last else SUB)
        return (2 * t + 2) * SUB

    B = lambda name, n, c: [Bar(f"{name}{i}", c) for i in range(n)]  # noqa: E731
    q_full, q_empty = B("q_full", NQB, 1), B("q_empty", NQB, 1)
    full, empty = B("full", NSLOT, 1), B("empty", NSLOT, 1)
    s_full, p_full, o_done = B("s_full", 2, 1), B("p_full", 2, 1), B("o_done", 2, 1)
    o_free = B("o_free", NOB, 1)
    u_full, u_empty = B("u_full", NU, 1), B("u_empty", NU, nprod + 2)
    ring = [None] * NU
    slot_pos, slot_landed, slot_readers = [None] * NSLOT, [False] * NSLOT, [0] * NSLOT
    q_unit, q_landed, q_readers = [None] * NQB, [False] * NQB, [0] * NQB
    o_epilogue = [False] * NOB
    copies, pipe = [], deque()
    s_read, p_written = set(), set()

    def wait(bar, parity, phase):
        while not bar.try_wait(parity):
            yield
        if bar.phase <= phase:
            raise StaleWait(f"{bar.name}: parity wait for phase {phase} passed with "
                            f"{bar.phase} phases complete")

    def take(k):
        yield from wait(u_full[k % NU], (k // NU) & 1, k // NU)
        kk, u = ring[k % NU]
        assert kk == k, "unit ring entry overwritten before it was read"
        return u

    def scheduler():
        itn = 0
        for k in range(len(units) + 1):
            if k >= NU:
                yield from wait(u_empty[k % NU], (k // NU - 1) & 1, k // NU - 1)
            u = units[k] if k < len(units) else None
            ring[k % NU] = (k, u)
            u_full[k % NU].arrive()
            if u is None:
                return
            if u["ntiles"]:
                qb = itn % NQB
                if itn >= NQB:
                    yield from wait(q_empty[qb], (itn // NQB - 1) & 1, itn // NQB - 1)
                assert not q_readers[qb], "Q buffer reloaded while MMAs read it"
                q_unit[qb], q_landed[qb] = itn, False
                q_full[qb].arrive(tx=1)
                copies.append((q_full[qb], "q", qb))
                itn += 1
            yield

    def producer(pw):
        seq = 0

        def group(nbytes):
            nonlocal seq
            for _ in range(SUB):
                if seq % nprod == pw:
                    s = seq % NSLOT
                    if seq >= NSLOT:
                        yield from wait(empty[s], (seq // NSLOT - 1) & 1, seq // NSLOT - 1)
                    assert not slot_readers[s], f"slot {s} re-armed while an MMA reads it"
                    slot_pos[s], slot_landed[s] = seq, nbytes == 0
                    full[s].arrive(tx=nbytes)
                    if nbytes:
                        copies.append((full[s], "kv", s))
                seq += 1
                yield

        prev, k = False, 0
        while True:
            u = yield from take(k)
            u_empty[k % NU].arrive()
            k += 1
            if u is None:
                break
            for j in range(u["ntiles"]):
                if PV_FIRST and order == "fixed" and j == 0 and prev:
                    yield from group(1)          # V(t - 1)
                    yield from group(1)          # K(t)
                else:
                    yield from group(1)          # K(t)
                    if prev:
                        yield from group(1)      # V(t - 1)
                prev = True
        if prev:
            if not (PV_FIRST and order == "fixed"):
                yield from group(0)              # empty K
            yield from group(1)                  # V(last)

    def mma_read(reads, q=None):
        for s, p in reads:
            assert slot_pos[s] == p and slot_landed[s], \
                f"MMA reads slot {s} for position {p}: holds {slot_pos[s]}"
            slot_readers[s] += 1
        if q is not None:
            assert q_landed[q[0]] and q_unit[q[0]] == q[1], "MMA reads a Q not landed"
            q_readers[q[0]] += 1
        pipe.append(("mma", reads, q))

    def mma():
        t = itn = k = 0
        pv = None

        def issue_pv(tp, cnt, ob, first, last, itn_p):
            if first and itn_p >= NOB:
                yield from wait(o_free[ob], (itn_p // NOB - 1) & 1, itn_p // NOB - 1)
                assert not o_epilogue[ob], "O overwritten during its epilogue"
            yield from wait(p_full[tp & 1], (tp >> 1) & 1, tp >> 1)
            assert tp in p_written
            p0 = pos_v(tp, last)
            for s in range(SUB):
                sl = (p0 + s) % NSLOT
                yield from wait(full[sl], ((p0 + s) // NSLOT) & 1, (p0 + s) // NSLOT)
                if s * (VKEYS // 16) < (cnt + 15) // 16:
                    mma_read([(sl, p0 + s)])
                pipe.append(("commit", empty[sl]))
            pipe.append(("commit", o_done[tp & 1]))

        while True:
            u = yield from take(k)
            u_empty[k % NU].arrive()
            k += 1
            if u is None:
                break
            if not u["ntiles"]:
                continue
            qb, ob = itn % NQB, itn % NOB
            if pv is not None and PV_FIRST and (
                    order == "fixed" or not q_full[qb].try_wait((itn // NQB) & 1)):
                yield from issue_pv(*pv)
                pv = None
            yield from wait(q_full[qb], (itn // NQB) & 1, itn // NQB)
            for j in range(u["ntiles"]):
                assert t < 2 or (t - 2) in s_read, "S overwritten before the softmax read it"
                p0 = pos_k(t, j == 0)
                for s in range(SUB):
                    sl = (p0 + s) % NSLOT
                    yield from wait(full[sl], ((p0 + s) // NSLOT) & 1, (p0 + s) // NSLOT)
                    mma_read([(sl, p0 + s)], (qb, itn))
                    pipe.append(("commit", empty[sl]))
                pipe.append(("commit", s_full[t & 1]))
                if j == u["ntiles"] - 1:
                    pipe.append(("commit", q_empty[qb]))
                if pv is not None:
                    yield from issue_pv(*pv)
                pv = (t, min(BN, u["kend"] - j * BN), ob, j == 0, j == u["ntiles"] - 1, itn)
                t += 1
                yield
            itn += 1
        if pv is not None:
            if not (PV_FIRST and order == "fixed"):
                p0 = pos_k(t, False)
                for s in range(SUB):
                    sl = (p0 + s) % NSLOT
                    yield from wait(full[sl], ((p0 + s) // NSLOT) & 1, (p0 + s) // NSLOT)
                    empty[sl].arrive()
            yield from issue_pv(*pv)

    def softmax():
        t = itn = k = 0
        while True:
            u = yield from take(k)
            u_empty[k % NU].arrive()
            k += 1
            if u is None:
                break
            for j in range(u["ntiles"]):
                yield from wait(s_full[t & 1], (t >> 1) & 1, t >> 1)
                s_read.add(t)
                cnt = min(BN, u["kend"] - j * BN)
                if cnt & 15:   # zero the value rows past the last key in the slot
                    pos = pos_v(t, j == u["ntiles"] - 1) + cnt // VKEYS
                    pv1 = pos_v(t - 1, j == 0) if t else 0
                    if t and pv1 <= pos - NSLOT < pv1 + SUB:
                        yield from wait(o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, (t - 1) >> 1)
                    sl = pos % NSLOT
                    yield from wait(full[sl], (pos // NSLOT) & 1, pos // NSLOT)
                    assert slot_pos[sl] == pos and slot_landed[sl] and not slot_readers[sl]
                p_written.add(t)
                p_full[t & 1].arrive()
                t += 1
                yield
            if u["ntiles"]:
                yield from wait(o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, (t - 1) >> 1)
                o_epilogue[itn % NOB] = True
                yield
                o_epilogue[itn % NOB] = False
                o_free[itn % NOB].arrive()
                itn += 1

    roles = [scheduler(), mma(), softmax()] + [producer(pw) for pw in range(nprod)]
    alive = list(range(len(roles)))
    for _ in range(3_000_000):
        if not (alive or copies or pipe):
            return
        c = rnd.randrange(len(alive) + bool(copies) + bool(pipe))
        if c < len(alive):
            try:
                next(roles[alive[c]])
            except StopIteration:
                alive.remove(alive[c])
        elif copies and c == len(alive):
            bar, kind, i = copies.pop(rnd.randrange(len(copies)))
            (q_landed if kind == "q" else slot_landed)[i] = True
            bar.complete_tx(1)
        else:
            item = pipe.popleft()
            if item[0] == "commit":
                item[1].arrive()
            else:
                for s, _ in item[1]:
                    slot_readers[s] -= 1
                if item[2] is not None:
                    q_readers[item[2][0]] -= 1
    raise AssertionError("no progress: the protocol deadlocked")


CASES = {
    # varlen causal prefill at head_dim 256, eight query heads per KV head
    "prefill-D256": (256, units_of([375, 434, 425, 441, 424, 446, 440, 435], 256, 8)),
    "ragged-D256": (256, units_of([60, 45, 130, 7, 300], 256, 8)),
    # prefill chunks and verify windows over prior context at head_dim 128
    "mixed-D128": (128, units_of([512, 512, 3, 5, 2], 128, 4, prior=[900, 1500, 800, 300, 2000])),
    "mixed-D64": (64, units_of([100, 37, 5], 64, 2, prior=[200, 0, 50])),
}


@pytest.mark.parametrize("nprod", [4, 6, 8])
@pytest.mark.parametrize("case", sorted(CASES))
def test_protocol_has_no_stale_wait_or_overwrite(case, nprod):
    D, units = CASES[case]
    for seed in range(25):
        order = list(units)
        random.Random(seed).shuffle(order)
        simulate(D, order[:48], nprod, seed)


def test_the_model_finds_the_earlier_claim_order_defect():
    """Issuing the previous unit's last PV first only when the new Q has not
    landed frees ring positions out of order; with producers far enough ahead
    a parity wait then passes on a phase still open."""
    D, units = CASES["prefill-D256"]
    found = False
    for seed in range(40):
        order = list(units)
        random.Random(seed).shuffle(order)
        try:
            simulate(D, order[:48], 6, seed, order="dynamic")
        except (StaleWait, AssertionError):
            found = True
            break
    assert found
