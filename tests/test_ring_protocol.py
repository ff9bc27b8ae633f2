"""A host-side model of the multi-query kernel's synchronisation protocol
(paged_prefill_tc_kernel in csrc/prefill_tc.cuh), run under random
interleavings.

The kernel's roles meet only through mbarriers whose waits test a phase
*parity*: a wait for phase k passes as soon as the barrier's current phase
has the other parity, so it cannot tell phase k from phase k - 2.  Whether
every wait is at most one phase away depends on the order in which the roles
fill and free the shared-memory rings of K and V sub-tiles, the unit ring,
the Q buffers, and the S/P and O regions of TMEM.  This model replays that
order with the kernel's arithmetic -- a K ring and a V ring of 16 KB
sub-tiles filled round robin by their producer warps, an S issuer and a PV
issuer (each frees its ring in fill order), NSB S/P buffers and NOB O
accumulators by head_dim, the softmax's zeroing of value rows past a tile's
last key -- and checks, for every interleaving it draws:

* no parity wait passes while the phase it waits for is still open;
* a slot is re-armed only after every MMA reading it has finished;
* every MMA reads a slot (or Q buffer) holding the sub-tile it expects, landed;
* S(t) does not overwrite P(t - NSB) before PV(t - NSB) has read it, and O is
  not overwritten during its epilogue.

The tensor pipe completes MMAs and commits in issue order; TMA copies land in
any order.  Two planted mistakes show that the model has teeth: dropping the
S issuer's wait for PV(t - NSB), and dropping the softmax's wait for the PV
that last read the slot it zeroes.
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


def simulate(D, units, kp, vp, seed, mutate=None):
    """One random interleaving of the kernel's roles over `units` (kp K and vp
    V producer warps); raises AssertionError on a violation."""
    rnd = random.Random(seed)
    SUB = D // 64
    NR = 5 if D >= 128 else 6            # slots per ring
    NQB = 1 if D >= 256 else 2
    NSB = 2 if D >= 256 else 3           # S/P buffers in TMEM
    NOB = 2 if D <= 64 else 1
    NU, BN = 8, 128
    VKEYS = BN // SUB
    B = lambda n, k, c: [Bar(f"{n}{i}", c) for i in range(k)]  # noqa: E731
    q_full, q_empty = B("q_full", NQB, 1), B("q_empty", NQB, 1)
    kfull, kempty = B("kfull", NR, 1), B("kempty", NR, 1)
    vfull, vempty = B("vfull", NR, 1), B("vempty", NR, 1)
    s_full, p_full, o_done = B("s_full", NSB, 1), B("p_full", NSB, 1), B("o_done", NSB, 1)
    o_free = B("o_free", NOB, 1)
    u_full, u_empty = B("u_full", NU, 1), B("u_empty", NU, 1 + kp + vp + 2)
    ring = [None] * NU
    kslot = {"pos": [None] * NR, "landed": [False] * NR, "readers": [0] * NR}
    vslot = {"pos": [None] * NR, "landed": [False] * NR, "readers": [0] * NR}
    q_unit, q_landed, q_readers = [None] * NQB, [False] * NQB, [0] * NQB
    o_epi = [False] * NOB
    s_buf_readers = [0] * 3   # PV MMAs in flight reading P from S buffer b
    copies, pipe = [], deque()
    state = {"s_read": set(), "p_written": set(), "s_written": set()}

    def wait(bar, parity, phase):
        while not bar.try_wait(parity):
            yield
        if bar.phase <= phase:
            raise StaleWait(f"{bar.name}: wait for phase {phase} passed at {bar.phase}")

    def take(k):
        yield from wait(u_full[k % NU], (k // NU) & 1, k // NU)
        kk, u = ring[k % NU]
        assert kk == k
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
                assert not q_readers[qb], "Q reloaded while read"
                q_unit[qb], q_landed[qb] = itn, False
                q_full[qb].arrive(tx=1)
                copies.append((q_full[qb], "q", qb))
                itn += 1
            yield

    def producer(which, pw, nw):
        full, empty, sl = (kfull, kempty, kslot) if which == "k" else (vfull, vempty, vslot)
        seq = 0
        k = 0
        while True:
            u = yield from take(k)
            u_empty[k % NU].arrive()
            k += 1
            if u is None:
                break
            for j in range(u["ntiles"]):
                for s in range(SUB):
                    if seq % nw == pw:
                        slot = seq % NR
                        if seq >= NR:
                            yield from wait(empty[slot], (seq // NR - 1) & 1, seq // NR - 1)
                        assert not sl["readers"][slot], f"{which} slot {slot} re-armed while read"
                        if which == "v" and zeroing[0] == slot:
                            raise AssertionError("V slot re-armed during zeroing")
                        sl["pos"][slot], sl["landed"][slot] = seq, False
                        full[slot].arrive(tx=1)
                        copies.append((full[slot], which, slot))
                    seq += 1
                    yield

    def read(sl, slot, pos, tag):
        assert sl["pos"][slot] == pos and sl["landed"][slot], \
            f"{tag}: slot {slot} holds {sl['pos'][slot]}, wants {pos}"
        sl["readers"][slot] += 1

    def mma_s():
        t = itn = k = 0
        while True:
            u = yield from take(k)
            u_empty[k % NU].arrive()
            k += 1
            if u is None:
                break
            if not u["ntiles"]:
                continue
            qb = itn % NQB
            yield from wait(q_full[qb], (itn // NQB) & 1, itn // NQB)
            for j in range(u["ntiles"]):
                b = t % NSB
                if t >= NSB and mutate != "no_sbuf_wait":
                    yield from wait(o_done[b], ((t - NSB) // NSB) & 1, (t - NSB) // NSB)
                if s_buf_readers[b]:
                    raise AssertionError(f"S({t}) overwrites P({t-NSB}) still read by PV")
                assert t < NSB or (t - NSB) in state["s_read"]
                reads = []
                for s in range(SUB):
                    p = t * SUB + s
                    slot = p % NR
                    yield from wait(kfull[slot], (p // NR) & 1, p // NR)
                for s in range(SUB):
                    p = t * SUB + s
                    read(kslot, p % NR, p, "S")
                    reads.append(("k", p % NR))
                assert q_landed[qb] and q_unit[qb] == itn
                q_readers[qb] += 1
                pipe.append(("mma", reads, ("q", qb), ("sw", b, t)))
                for s in range(SUB):
                    pipe.append(("commit", kempty[(t * SUB + s) % NR]))
                pipe.append(("commit", s_full[b]))
                if j == u["ntiles"] - 1:
                    pipe.append(("commit", q_empty[qb]))
                t += 1
                yield
            itn += 1

    def mma_pv():
        t = itn = k = 0
        while True:
            u = yield from take(k)
            u_empty[k % NU].arrive()
            k += 1
            if u is None:
                break
            if not u["ntiles"]:
                continue
            ob = itn % NOB
            for j in range(u["ntiles"]):
                if j == 0 and itn >= NOB:
                    yield from wait(o_free[ob], (itn // NOB - 1) & 1, itn // NOB - 1)
                    assert not o_epi[ob], "O overwritten during its epilogue"
                yield from wait(p_full[t % NSB], (t // NSB) & 1, t // NSB)
                assert t in state["p_written"]
                cnt = min(BN, u["kend"] - j * BN)
                nk = (cnt + 15) // 16
                for s in range(SUB):
                    p = t * SUB + s
                    yield from wait(vfull[p % NR], (p // NR) & 1, p // NR)
                reads = []
                for s in range(SUB):
                    p = t * SUB + s
                    if s * (VKEYS // 16) < nk:
                        read(vslot, p % NR, p, "PV")
                        reads.append(("v", p % NR))
                s_buf_readers[t % NSB] += 1
                pipe.append(("mma", reads, None, ("pr", t % NSB, t)))
                for s in range(SUB):
                    pipe.append(("commit", vempty[(t * SUB + s) % NR]))
                pipe.append(("commit", o_done[t % NSB]))
                t += 1
                yield
            itn += 1

    zeroing = [None]

    def softmax():
        t = itn = k = 0
        while True:
            u = yield from take(k)
            u_empty[k % NU].arrive()
            k += 1
            if u is None:
                break
            for j in range(u["ntiles"]):
                yield from wait(s_full[t % NSB], (t // NSB) & 1, t // NSB)
                assert t in state["s_written"]
                state["s_read"].add(t)
                cnt = min(BN, u["kend"] - j * BN)
                if cnt & 15:
                    pos = t * SUB + cnt // VKEYS
                    prev = pos - NR
                    tp = prev // SUB if prev >= 0 else -1   # tile of the slot's previous sub-tile
                    if tp >= 0 and tp > t - NSB and mutate != "no_vtail_wait":
                        yield from wait(o_done[tp % NSB], (tp // NSB) & 1, tp // NSB)
                    slot = pos % NR
                    yield from wait(vfull[slot], (pos // NR) & 1, pos // NR)
                    assert vslot["pos"][slot] == pos and vslot["landed"][slot] \
                        and not vslot["readers"][slot], "V-tail zeroing on a wrong or busy slot"
                    zeroing[0] = slot
                    yield
                    zeroing[0] = None
                state["p_written"].add(t)
                p_full[t % NSB].arrive()
                t += 1
                yield
            if u["ntiles"]:
                yield from wait(o_done[(t - 1) % NSB], ((t - 1) // NSB) & 1, (t - 1) // NSB)
                ob = itn % NOB
                o_epi[ob] = True
                yield
                o_epi[ob] = False
                o_free[ob].arrive()
                itn += 1

    roles = [scheduler(), mma_s(), mma_pv(), softmax()]
    roles += [producer("k", i, kp) for i in range(kp)] + [producer("v", i, vp) for i in range(vp)]
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
            {"q": q_landed, "k": kslot["landed"], "v": vslot["landed"]}[kind][i] = True
            bar.complete_tx(1)
        else:
            # the tensor pipe executes in order; two issuers' MMAs interleave in the pipe
            item = pipe.popleft()
            if item[0] == "commit":
                item[1].arrive()
            else:
                for which, slot in item[1]:
                    (kslot if which == "k" else vslot)["readers"][slot] -= 1
                if item[2]:
                    q_readers[item[2][1]] -= 1
                tag = item[3]
                if tag[0] == "sw":
                    state["s_written"].add(tag[2])
                if tag[0] == "pr":
                    s_buf_readers[tag[1]] -= 1
    raise AssertionError("deadlock")


CASES = {
    # varlen causal prefill at head_dim 256, eight query heads per KV head
    "prefill-D256": (256, units_of([375, 434, 425, 441, 424, 446, 440, 435], 256, 8)),
    "ragged-D256": (256, units_of([60, 45, 130, 7, 300], 256, 8)),
    # prefill chunks and verify windows over prior context at head_dim 128
    "mixed-D128": (128, units_of([512, 512, 3, 5, 2], 128, 4, prior=[900, 1500, 800, 300, 2000])),
    "mixed-D64": (64, units_of([100, 37, 5], 64, 2, prior=[200, 0, 50])),
    "noncausal-D128": (128, units_of([40, 3, 77], 128, 8, prior=[300, 10, 0], causal=False)),
}


def _run(case, kp, vp, seeds, mutate=None):
    D, units = CASES[case]
    for seed in seeds:
        order = list(units)
        random.Random(seed).shuffle(order)
        simulate(D, order[:48], kp, vp, seed, mutate=mutate)


@pytest.mark.parametrize("kp,vp", [(2, 2), (1, 1), (3, 3)])
@pytest.mark.parametrize("case", sorted(CASES))
def test_protocol_has_no_stale_wait_or_overwrite(case, kp, vp):
    _run(case, kp, vp, range(20))


@pytest.mark.parametrize("mutate,case,seeds", [
    ("no_sbuf_wait", "prefill-D256", range(20)),
    ("no_vtail_wait", "ragged-D256", range(200)),
])
def test_the_model_finds_planted_mistakes(mutate, case, seeds):
    with pytest.raises(AssertionError):
        _run(case, 2, 2, seeds, mutate=mutate)
