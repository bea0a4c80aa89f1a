"""Barrier-level model of the bf16 attention kernel's pipeline (attn_tc.cu), run on the CPU.

The model follows the kernel's schedule exactly: the same work items and tile sequences
(make_item / make_half / half_next), the producer's K/V ring of NS slots with one FULL
barrier per tile on its K slot, the issuer's S-after-PV order per half, its per-slot
pending-S counts, QFULL/QFREE, PFULL, PVDONE and OFREE, and the rule that a half's S on a
tile more than two tiles ahead is held back until the loop is two tiles short of it.
Barriers complete phases; every wait names the phase it expects, so a wait that would
pass on a stale or a future phase fails the test.  The processes are interleaved in
seeded random order until all finish; a state in which none can move is a deadlock.

It pins the property the GPU tests can only sample: no shape deadlocks, including the
group-aligned window with groups of more than 128 tokens, where half B's band starts
several tiles after its last core tile."""
import os
import random
import re

import pytest

BM = BN = 128
NS = 5

KERNEL = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "sparse_long_context_cca_gb300",
                      "csrc", "attn_tc.cu")


def test_model_constants_match_the_kernel():
    """The model's tile sizes and ring depth are the kernel's: a change there must be
    carried into the model before it can say anything about the new pipeline."""
    src = open(KERNEL).read()
    found = {name: int(v) for name, v in re.findall(r"constexpr int (BM|BN|NS) = (\d+);", src)}
    assert found == {"BM": BM, "BN": BN, "NS": NS}, found


def lo_of(i, w):
    return max(0, i - w + 1)


def win_of(i, w, g, wm):
    lo = lo_of(i, w)
    return (lo // g) * g if wm else lo


class Item:
    def __init__(self, N, g, w, wm, k, BH, n_pairs, q_off=0, n_q=None):
        # rows [q_off, q_off + n_q) of the N-token sequence (the whole of it by default)
        n_q = N - q_off if n_q is None else n_q
        pair = n_pairs - 1 - k // BH
        i0 = q_off + pair * 2 * BM
        self.lo0 = win_of(i0, w, g, wm)
        self.valid, self.tc, self.kl, self.kh = [], [], [], []
        last = None
        for a in (i0, i0 + BM):
            if a - q_off >= n_q:
                self.valid.append(False)
                self.tc.append(0), self.kl.append(0), self.kh.append(0)
                continue
            b = min(a + BM - 1, q_off + n_q - 1)
            last = b
            self.valid.append(True)
            self.tc.append((lo_of(b, w) // g + BN - 1) // BN)
            self.kl.append((win_of(a, w, g, wm) - self.lo0) // BN)
            self.kh.append((b - self.lo0) // BN + 1)
        self.Tc = max(self.tc)
        self.T = self.Tc + (last - self.lo0) // BN + 1

    def uses(self, h, t):
        if not self.valid[h]:
            return False
        if t < self.Tc:
            return t < self.tc[h]
        return self.kl[h] <= t - self.Tc < self.kh[h]

    def first(self, h):
        return 0 if self.tc[h] > 0 else self.Tc + self.kl[h]

    def next(self, h, t):
        if t < self.Tc:
            return t + 1 if t + 1 < self.tc[h] else self.Tc + self.kl[h]
        return t + 1 if t + 1 < self.Tc + self.kh[h] else -1

    def count(self, h):
        return self.tc[h] + self.kh[h] - self.kl[h] if self.valid[h] else 0

    def max_step(self, h):
        return self.Tc + self.kl[h] - (self.tc[h] - 1) if self.valid[h] and self.tc[h] > 0 else 1


class Bar:
    def __init__(self, name):
        self.name, self.phases = name, 0

    def arrive(self):
        self.phases += 1


def run(N, g, w, wm, grid, blk, seed, H=2, q_off=0, n_q=None):
    """Runs the model for CTA `blk` of `grid`; returns None, or the blocked waits on deadlock.
    q_off, n_q: a launch over the rows [q_off, q_off + n_q) only (cca_attn_fwd_rows)."""
    n_rows = N - q_off if n_q is None else n_q
    n_pairs = (n_rows + 2 * BM - 1) // (2 * BM)
    items = [Item(N, g, w, wm, k, H, n_pairs, q_off, n_rows) for k in range(blk, n_pairs * H, grid)]
    qfull, qfree = Bar("qfull"), Bar("qfree")
    full = [Bar(f"full{s}") for s in range(NS)]
    empty = [Bar(f"empty{s}") for s in range(NS)]
    sfull, pfull = [Bar("sfullA"), Bar("sfullB")], [Bar("pfullA"), Bar("pfullB")]
    pvdone, ofree = [Bar("pvdoneA"), Bar("pvdoneB")], [Bar("ofreeA"), Bar("ofreeB")]

    def W(bar, phase):  # wait until `bar` has completed `phase` phases; never more than one ahead
        return (bar, phase)

    # data flow: which global tile each ring slot holds (and whether its readers are done),
    # which (item, tile) each half's pending S holds, and which item's Q is loaded
    slot_tile = [None] * NS
    s_queue = [[], []]
    q_item = [None]

    def producer():
        u = 0
        for n, it in enumerate(items):
            yield W(qfree, n)          # the previous item's Q buffer is free
            q_item[0] = n
            qfull.arrive()
            for _ in range(it.T):
                ks, vs = u % NS, (u + 1) % NS
                yield W(empty[ks], u // NS)      # slot's previous use released
                yield W(empty[vs], (u + 1) // NS)
                slot_tile[ks] = ("K", u // 2)
                slot_tile[vs] = ("V", u // 2)
                full[ks].arrive()                 # K and V of the tile on the K slot
                u += 2

    def issuer():
        ubase, pend, pf, nh = 0, [0] * NS, [0, 0], [0, 0]
        for n, it in enumerate(items):
            yield W(qfull, n + 1)
            assert q_item[0] == n, ("Q", q_item[0], n)
            s_left = [it.count(0) + it.count(1)]

            def issue_s(h, t):
                uk = ubase + 2 * t
                slot = uk % NS
                if pend[slot] == 0:
                    yield W(full[slot], uk // (2 * NS) + 1)
                    pend[slot] = int(it.uses(0, t)) + int(it.uses(1, t))
                assert it.uses(h, t) and pend[slot] > 0
                assert slot_tile[slot] == ("K", uk // 2), ("K slot", slot_tile[slot], uk // 2)
                assert slot_tile[(uk + 1) % NS] == ("V", uk // 2), ("V slot", slot_tile[(uk + 1) % NS], uk // 2)
                assert q_item[0] == n, ("Q overwritten", q_item[0], n)
                s_queue[h].append((n, t))
                sfull[h].arrive()
                pend[slot] -= 1
                if pend[slot] == 0:
                    empty[slot].arrive()
                s_left[0] -= 1
                if s_left[0] == 0:
                    qfree.arrive()

            b_first = it.valid[1] and it.first(1) < it.first(0)
            for q in range(2):
                h = 1 - q if b_first else q
                if it.valid[h]:
                    yield from issue_s(h, it.first(h))
            needs_defer = max(it.max_step(0), it.max_step(1)) > 2
            first_pv, defer = [True, True], [-1, -1]
            for t in range(it.T):
                vslot = (ubase + 2 * t + 1) % NS
                for h in range(2):
                    if defer[h] >= 0 and defer[h] <= t + 2:
                        yield from issue_s(h, defer[h])
                        defer[h] = -1
                for h in range(2):
                    if not it.uses(h, t):
                        continue
                    yield W(pfull[h], pf[h] + 1)
                    pf[h] += 1
                    assert slot_tile[vslot] == ("V", (ubase + 2 * t) // 2), ("V at PV", slot_tile[vslot], t)
                    if first_pv[h]:
                        yield W(ofree[h], nh[h])
                    first_pv[h] = False
                    tn = it.next(h, t)
                    if tn > t + 2:
                        # only items that take the deferring copy of the loop ever get here
                        assert needs_defer, (N, g, w, wm, t, tn)
                        defer[h] = tn
                    elif tn >= 0:
                        yield from issue_s(h, tn)
                    else:
                        pvdone[h].arrive()
                empty[vslot].arrive()
            assert defer == [-1, -1]
            ubase += 2 * it.T
            for h in range(2):
                nh[h] += int(it.valid[h])

    def softmax(h):
        seen, done = 0, 0
        for n, it in enumerate(items):
            if not it.valid[h]:
                continue
            t, order = it.first(h), []
            while t >= 0:
                yield W(sfull[h], seen + 1)
                seen += 1
                assert s_queue[h] and s_queue[h][0] == (n, t), ("S", h, s_queue[h][:1], (n, t))
                s_queue[h].pop(0)
                order.append(t)
                pfull[h].arrive()
                t = it.next(h, t)
            assert order == [x for x in range(it.T) if it.uses(h, x)]
            yield W(pvdone[h], done + 1)
            ofree[h].arrive()
            done += 1

    procs = {"producer": producer(), "issuer": issuer(), "softmaxA": softmax(0), "softmaxB": softmax(1)}
    waiting = dict.fromkeys(procs)
    rng = random.Random(seed)
    while procs:
        moved = False
        for name in rng.sample(sorted(procs), len(procs)):
            for _ in range(rng.randint(1, 4)):
                wt = waiting[name]
                if wt is not None:
                    bar, phase = wt
                    if bar.phases < phase:
                        break
                    # an mbarrier only tells its current phase's parity: a wait may not run
                    # more than one phase behind the barrier
                    assert bar.phases <= phase + 1, (name, bar.name, bar.phases, phase)
                    waiting[name] = None
                    moved = True
                try:
                    waiting[name] = next(procs[name])
                    moved = True
                except StopIteration:
                    del procs[name]
                    waiting.pop(name)
                    break
        if not moved:
            return {n: waiting[n][0].name for n in procs if waiting[n] is not None}
    return None


SHAPES = [(N, g, w, wm)
          for wm in (0, 1)
          for N in (128, 640, 1024, 2048, 4096)
          for g in (1, 3, 16, 64, 128, 256, 384, 512, 1024)
          if N % g == 0
          for w in (1, 4, 96, 300, 1024, 5000)]


@pytest.mark.parametrize("wm", [0, 1])
def test_no_deadlock_and_phases_consistent(wm):
    bad = []
    for N, g, w, m in SHAPES:
        if m != wm:
            continue
        for grid, blk in ((1, 0), (2, 1), (5, 0)):
            r = run(N, g, w, m, grid, blk, seed=N * 7 + g * 3 + w + grid)
            if r is not None:
                bad.append(((N, g, w, m, grid, blk), r))
    assert not bad, bad[:3]


def test_large_groups_take_the_deferring_loop():
    """With the group-aligned window and g = 512, half B's band starts four tiles after its
    core tile: the item needs the deferring copy of the loop, and the model completes."""
    n_pairs = 4096 // 256
    items = [Item(4096, 512, 4, 1, k, 2, n_pairs) for k in range(n_pairs * 2)]
    assert any(max(it.max_step(0), it.max_step(1)) > 2 for it in items)
    assert run(4096, 512, 4, 1, 1, 0, seed=1) is None


RANGES = [(N, g, w, wm, q_off, n_q)
          for wm in (0, 1)
          for N, g in ((2048, 16), (4096, 512), (3072, 384), (1024, 1))
          for w in (1, 96, 300, 1024)
          for q_off, n_q in ((16, 1000), (112, N - 112), (N // 2 - g, 300), (N - 1, 1), (0, 257))
          if q_off >= 0 and q_off + n_q <= N]


@pytest.mark.parametrize("wm", [0, 1])
def test_row_ranges_do_not_deadlock(wm):
    """Launches over a row range (a shard of a sequence) deal items of 256 rows from q_off, so
    their tile sequences start at other offsets than the whole sequence's: the same model,
    the same property."""
    bad = []
    deferring = 0
    for N, g, w, m, q_off, n_q in RANGES:
        if m != wm:
            continue
        n_pairs = (n_q + 2 * BM - 1) // (2 * BM)
        deferring += sum(max(it.max_step(0), it.max_step(1)) > 2
                         for it in (Item(N, g, w, m, k, 2, n_pairs, q_off, n_q) for k in range(2 * n_pairs)))
        n_items = 2 * ((n_q + 2 * BM - 1) // (2 * BM))  # two heads
        for grid, blk in ((1, 0), (3, 2)):
            if blk >= n_items:  # the kernel launches min(items, SMs) CTAs
                continue
            r = run(N, g, w, m, grid, blk, seed=N + q_off * 5 + w, q_off=q_off, n_q=n_q)
            if r is not None:
                bad.append(((N, g, w, m, q_off, n_q, grid, blk), r))
    assert not bad, bad[:3]
    if wm == 1:
        assert deferring > 0  # the group-aligned window with large groups takes the deferring loop
