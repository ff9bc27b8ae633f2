"""A host-side model of the quantised-cache decode kernel's synchronisation
protocol (paged_decode_tc_fp8_kernel in csrc/decode_tc_fp8.cuh), run under
random interleavings.

Its roles meet through mbarriers whose waits test a phase parity, so a wait
cannot tell phase k from phase k - 2; whether every wait stays within one
phase depends on the order in which the roles fill and free their buffers.
The model replays that order -- the K-code ring (freed by the S MMAs) and the
V-code ring (freed by the converters) filled by two producer warps each, the
f16 V stages (freed by the PV MMAs), the scale ring (cp.async copies landing
in any order, freed by the softmax), the two bf16 Q buffers and two E4M3 Q
buffers of the query warp with the ring of four 2^-e factors, two S buffers,
two P buffers, two O accumulators written out one item late, and the lazy O
rescale -- and checks, for every interleaving it draws:

* no parity wait passes while the phase it waits for is still open;
* no buffer is rewritten while an MMA, a converter or the softmax still reads
  it, and every read finds the tile (or item) it expects, landed;
* an item's O accumulator is read after its last PV and before the first PV
  of the item after next overwrites it.

The tensor pipe completes MMAs and commits in issue order; TMA and cp.async
copies land in any order.  Five planted mistakes show that the model has
teeth: a scale warp that does not wait for the softmax to free a stage,
converters that do not wait for the PV MMAs, K producers that do not wait for
the S MMAs, a query warp that does not wait for the S MMAs of the item before
last, and outputs written two items late.  (Two of the kernel's waits -- the S
MMAs' wait for the softmax to free an S buffer, the softmax's wait for the PV
that last read a P buffer -- are implied by the MMA issue order, and leaving
them out breaks nothing here.)
"""
import random
from collections import deque

import pytest

from test_ring_protocol import Bar, StaleWait


def simulate(items, KS, seed, NRC=3, NRV=3, NSC=3, mutate=None):
    """One random interleaving over `items` (key tiles per item; 0 = an item
    without keys); raises AssertionError on a violation."""
    rnd = random.Random(seed)
    PW = 2   # producer warps per code ring
    B = lambda n, k, c: [Bar(f"{n}{i}", c) for i in range(k)]  # noqa: E731
    kc_full, kc_empty = B("kc_full", NRC, PW), B("kc_empty", NRC, 1)
    vc_full, vc_empty = B("vc_full", NRC, PW), B("vc_empty", NRC, 1)
    v_full, v_empty = B("v_full", NRV, 1), B("v_empty", NRV, 1)
    sc_full, sc_empty = B("sc_full", NSC, 1), B("sc_empty", NSC, 1)
    q_full, q8_full, q_empty = B("q_full", 2, 1), B("q8_full", 2, 1), B("q_empty", 2, 1)
    s_full, s_free = B("s_full", 2, 1), B("s_free", 2, 1)
    p_full, o_done, o_full = B("p_full", 2, 1), B("o_done", 2, 1), B("o_full", 2, 1)
    # buffer states: what each holds, whether it landed, who reads it now
    kc = [{"pos": None, "landed": False, "readers": 0} for _ in range(NRC)]
    vc = [{"pos": None, "landed": False, "reading": False} for _ in range(NRC)]
    vs = [{"pos": None, "readers": 0} for _ in range(NRV)]
    sc = [{"pos": None, "landed": 0} for _ in range(NSC)]
    qb16 = [{"item": None, "landed": False, "reading": False} for _ in range(2)]
    q8 = [{"item": None, "readers": 0} for _ in range(2)]
    q_inv = [None] * 4
    sbuf = [{"tile": None} for _ in range(2)]
    pbuf = [{"tile": None, "readers": 0} for _ in range(2)]
    obuf = [{"item": None, "last_pv": None, "pv_in_flight": 0} for _ in range(2)]
    copies, pipe = [], deque()
    tiles = [(i, j) for i, n in enumerate(items) for j in range(n)]   # non-empty items' tiles
    nz = [i for i, n in enumerate(items) if n]                        # items with tiles
    itn_of = {i: k for k, i in enumerate(nz)}
    last_tile_of = {}
    for g, (i, j) in enumerate(tiles):
        last_tile_of[i] = g

    def wait(bar, parity, phase):
        while not bar.try_wait(parity):
            yield
        if bar.phase <= phase:
            raise StaleWait(f"{bar.name}: wait for phase {phase} passed at {bar.phase}")

    def producer(which, pw):
        full, empty, ring = (kc_full, kc_empty, kc) if which == "k" else (vc_full, vc_empty, vc)
        for t in range(len(tiles)):
            for c in range(KS):
                idx = t * KS + c
                slot = idx % NRC
                if idx >= NRC and not (which == "k" and mutate == "no_kc_empty"):
                    yield from wait(empty[slot], (idx // NRC - 1) & 1, idx // NRC - 1)
                if which == "k":
                    assert not ring[slot]["readers"], f"K stage {slot} re-armed while read"
                else:
                    assert not ring[slot]["reading"], f"V-code stage {slot} re-armed while read"
                if pw == 0:
                    ring[slot]["pos"], ring[slot]["landed"] = idx, False
                full[slot].arrive(tx=1)
                copies.append((full[slot], which, slot))
                yield

    def scale_warp():
        for t in range(len(tiles)):
            s = t % NSC
            if t >= NSC and mutate != "no_sc_empty":
                yield from wait(sc_empty[s], (t // NSC - 1) & 1, t // NSC - 1)
            sc[s]["pos"], sc[s]["landed"] = t, 0
            copies.append((sc_full[s], "sc", s))   # lands, then the lane's arrival counts
            yield

    def query_warp():
        for k, i in enumerate(nz):
            b = k & 1
            if k >= 2 and mutate != "no_q_empty":
                yield from wait(q_empty[b], (k // 2 - 1) & 1, k // 2 - 1)
            assert not qb16[b]["reading"], "bf16 Q reloaded while read"
            qb16[b]["item"], qb16[b]["landed"] = k, False
            q_full[b].arrive(tx=1)
            copies.append((q_full[b], "q", b))
            yield from wait(q_full[b], (k // 2) & 1, k // 2)
            assert qb16[b]["landed"] and qb16[b]["item"] == k
            qb16[b]["reading"] = True
            yield
            assert not q8[b]["readers"], "E4M3 Q rewritten while S MMAs read it"
            q8[b]["item"] = k
            q_inv[k & 3] = k
            qb16[b]["reading"] = False
            q8_full[b].arrive()
            yield

    def converters():
        for t in range(len(tiles)):
            for c in range(KS):
                idx = t * KS + c
                cs, vsl = idx % NRC, idx % NRV
                yield from wait(vc_full[cs], (idx // NRC) & 1, idx // NRC)
                if idx >= NRV and mutate != "no_v_empty":
                    yield from wait(v_empty[vsl], (idx // NRV - 1) & 1, idx // NRV - 1)
                assert vc[cs]["pos"] == idx and vc[cs]["landed"], "converter reads a wrong stage"
                assert not vs[vsl]["readers"], f"f16 V stage {vsl} rewritten while PV reads it"
                vc[cs]["reading"] = True
                yield
                vs[vsl]["pos"] = idx
                vc[cs]["reading"] = False
                vc_empty[cs].arrive()
                v_full[vsl].arrive()
                yield

    def mma():
        gt = 0
        pend = None

        def issue_pv(g, first, last):
            i, _ = tiles[g]
            ob = itn_of[i] & 1
            yield from wait(p_full[g & 1], (g >> 1) & 1, g >> 1)
            assert pbuf[g & 1]["tile"] == g, "PV reads a wrong P"
            for c in range(KS):
                idx = g * KS + c
                yield from wait(v_full[idx % NRV], (idx // NRV) & 1, idx // NRV)
                assert vs[idx % NRV]["pos"] == idx, "PV reads a wrong V stage"
            if first:
                assert obuf[ob]["item"] is None or obuf[ob]["item"] == "read", \
                    f"first PV of item {i} overwrites an O not written out yet"
                obuf[ob]["item"] = i
            reads = [("v", (g * KS + c) % NRV) for c in range(KS)] + [("p", g & 1)]
            for kind, s in reads:
                (vs if kind == "v" else pbuf)[s]["readers"] += 1
            obuf[ob]["pv_in_flight"] += 1
            pipe.append(("mma", reads, ("o", ob, g if last else None)))
            pipe.append(("commit", o_done[g & 1]))
            for c in range(KS):
                pipe.append(("commit", v_empty[(g * KS + c) % NRV]))
            if last:
                pipe.append(("commit", o_full[ob]))

        for k, i in enumerate(nz):
            b = k & 1
            yield from wait(q8_full[b], (k // 2) & 1, k // 2)
            assert q8[b]["item"] == k, "S reads a wrong E4M3 Q"
            for j in range(items[i]):
                sb = gt & 1
                # (also implied by the PV order: PV(gt - 2) waited for P(gt - 2))
                if gt >= 2:
                    yield from wait(s_free[sb], (gt // 2 - 1) & 1, gt // 2 - 1)
                for c in range(KS):
                    idx = gt * KS + c
                    yield from wait(kc_full[idx % NRC], (idx // NRC) & 1, idx // NRC)
                    assert kc[idx % NRC]["pos"] == idx and kc[idx % NRC]["landed"]
                reads = [("k", (gt * KS + c) % NRC) for c in range(KS)]
                for _, s in reads:
                    kc[s]["readers"] += 1
                q8[b]["readers"] += 1
                pipe.append(("mma", reads + [("q8", b)], ("s", sb, gt)))
                pipe.append(("commit", s_full[sb]))
                for c in range(KS):
                    pipe.append(("commit", kc_empty[(gt * KS + c) % NRC]))
                if j == items[i] - 1:
                    pipe.append(("commit", q_empty[b]))
                if pend is not None:
                    yield from issue_pv(*pend)
                pend = (gt, j == 0, j == items[i] - 1)
                gt += 1
                yield
        if pend is not None:
            yield from issue_pv(*pend)

    def softmax():
        gt = 0

        def finish(item_itn):
            i, k = item_itn
            if k is None:
                return
            ob = k & 1
            yield from wait(o_full[ob], (k // 2) & 1, k // 2)
            assert obuf[ob]["item"] == i and obuf[ob]["last_pv"] == last_tile_of[i] \
                and not obuf[ob]["pv_in_flight"], f"item {i}'s output read before its last PV"
            obuf[ob]["item"] = "read"

        keep = 2 if mutate == "late_finish" else 1   # outputs pending after a first tile
        pending = deque()
        for i, n in enumerate(items):
            k = itn_of.get(i)
            for j in range(n):
                sb = gt & 1
                yield from wait(s_full[sb], (gt >> 1) & 1, gt >> 1)
                assert sbuf[sb]["tile"] == gt, "softmax reads a wrong S"
                s_free[sb].arrive()
                if j == 0:
                    assert q_inv[k & 3] == k, "softmax reads another item's 2^-e"
                s = gt % NSC
                yield from wait(sc_full[s], (gt // NSC) & 1, gt // NSC)
                assert sc[s]["pos"] == gt and sc[s]["landed"], "softmax reads wrong scales"
                sc_empty[s].arrive()
                if j >= 1 and rnd.random() < 0.3:   # a lazy O rescale
                    yield from wait(o_done[(gt - 1) & 1], ((gt - 1) >> 1) & 1, (gt - 1) >> 1)
                    assert not obuf[k & 1]["pv_in_flight"], "O rescaled while a PV writes it"
                pb = gt & 1
                # (redundant under in-order completion: S(gt) follows PV(gt - 2))
                if gt >= 2:
                    yield from wait(o_done[pb], ((gt >> 1) - 1) & 1, (gt >> 1) - 1)
                assert not pbuf[pb]["readers"], "P rewritten while PV reads it"
                pbuf[pb]["tile"] = gt
                p_full[pb].arrive()
                gt += 1
                yield
                while len(pending) >= keep:
                    yield from finish(pending.popleft())
            while len(pending) >= keep:   # an item without tiles
                yield from finish(pending.popleft())
            pending.append((i, k))
            yield
        while pending:
            yield from finish(pending.popleft())

    roles = [producer("k", 0), producer("k", 1), producer("v", 0), producer("v", 1),
             scale_warp(), query_warp(), converters(), mma(), softmax()]
    alive = list(range(len(roles)))
    for _ in range(2_000_000):
        if not (alive or copies or pipe):
            return
        c = rnd.randrange(len(alive) + bool(copies) + bool(pipe))
        if c < len(alive):
            try:
                next(roles[alive[c]])
            except StopIteration:
                alive.remove(alive[c])
        elif copies and c == len(alive):
            bar, kind, s = copies.pop(rnd.randrange(len(copies)))
            if kind == "k":
                kc[s]["landed"] = True
            elif kind == "v":
                vc[s]["landed"] = True
            elif kind == "q":
                qb16[s]["landed"] = True
            if kind == "sc":
                sc[s]["landed"] = 1
                bar.arrive()
            else:
                bar.complete_tx(1)
        else:
            item = pipe.popleft()
            if item[0] == "commit":
                item[1].arrive()
                continue
            for kind, s in item[1]:
                if kind == "k":
                    kc[s]["readers"] -= 1
                elif kind == "v":
                    vs[s]["readers"] -= 1
                elif kind == "p":
                    pbuf[s]["readers"] -= 1
                elif kind == "q8":
                    q8[s]["readers"] -= 1
            tag = item[2]
            if tag[0] == "s":
                sbuf[tag[1]]["tile"] = tag[2]
            else:
                ob = tag[1]
                obuf[ob]["pv_in_flight"] -= 1
                if tag[2] is not None:
                    obuf[ob]["last_pv"] = tag[2]
    raise AssertionError("deadlock")


CASES = {
    # the GQA decode batch's shape: items of up to four 128-key tiles
    "decode-D128": ([4, 4, 3, 1, 4, 2, 4, 4, 1, 3, 4, 4], 1),
    # long partitions at head_dim 256 (two 128-dim chunks per tile)
    "long-D256": ([8, 8, 5, 8, 2, 8], 2),
    # single-tile items and items without keys
    "ragged": ([1, 0, 1, 1, 0, 0, 2, 1, 1, 3, 0, 1], 1),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_protocol_has_no_stale_wait_or_overwrite(case):
    items, KS = CASES[case]
    for seed in range(40):
        # the kernel's stage counts: 4 code + 2 f16 V stages at head_dim 128, 3 + 2 at 256
        simulate(items, KS, seed, NRC=4 if KS == 1 else 3, NRV=2)


@pytest.mark.parametrize("mutate", ["no_sc_empty", "no_v_empty", "no_kc_empty", "no_q_empty",
                                    "late_finish"])
def test_the_model_finds_planted_mistakes(mutate):
    items, KS = CASES["decode-D128"]
    with pytest.raises(AssertionError):
        for seed in range(200):
            simulate(items, KS, seed, mutate=mutate)
