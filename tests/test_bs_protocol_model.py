"""A host model of the block-scaled kernel's barrier protocol (gemm_blockscale.cuh), run under
random interleavings: the TMA producer, the two MMA issuers and the eight accumulating warps
as coroutines over modelled mbarriers (a phase count; a parity wait passes once the phase of
that parity has completed), with the issuers' commits completing late, in each issuer's issue
order.  Every operand-stage read checks that the stage holds the k-tile the reader expects,
and every partial read that the buffer holds the pair and k-block the epilogue expects.

The kernel's protocol: the k-blocks of each work item pair up from its first (an odd last one
alone); pair q uses slot q % 2 (two TMEM buffers); issuer r issues the k-blocks whose index over
all of the CTA's items has parity r, each into the buffer of its position in the pair, after
waiting PEMPTY of the slot, and commits PFULL (counting two) or, for a lone k-block of the other
issuer, only arrives; an issuer waits FULL of each stage its k-blocks read and commits EMPTY after
the last of them (EMPTY counts one reader at 128-wide k-blocks, two below).

Two earlier forms are kept as negative controls, to show that the model catches the hazard
they had: a parity wait meeting a stage two phases on at small rings."""
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.phase = count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, parity):
        return (self.phase & 1) != parity


class Stale(AssertionError):
    pass


def run(items, bk, stages, seed, form="current"):
    """One interleaving of the protocol over work items of items[i] k-tiles each."""
    per_atom = 128 // bk
    rng = random.Random(seed)
    if form == "current":
        readers = 1 if bk == 128 else 2
    else:   # the alternate-pairs form: one issuer per pair
        readers = 2 if bk == 32 else 1
    FULL = [Bar(1) for _ in range(stages)]
    EMPTY = [Bar(readers) for _ in range(stages)]
    PFULL = [Bar(2 if form in ("current", "item_local") else 1) for _ in range(2)]
    PEMPTY = [Bar(8) for _ in range(2)]
    stage_tag, buf_tag = [None] * stages, [None] * 4
    pending = []   # commits in flight: (issuer, barrier)

    def producer():
        t, st, ph = 0, 0, 0
        for kc in items:
            for _ in range(kc):
                while not EMPTY[st].done(ph ^ 1):
                    yield
                stage_tag[st] = t
                FULL[st].arrive()
                t, st = t + 1, st + 1
                if st == stages:
                    st, ph = 0, ph ^ 1

    def issuer(r):
        kt_cur, st, ph, q0, kt_item, kbase = 0, 0, 0, 0, 0, 0
        for kc in items:
            nkb = kc * per_atom
            npairs = (nkb + 1) // 2
            if form == "alternate_pairs":
                pairs = range((q0 + r) & 1, npairs, 2)
            else:
                pairs = range(npairs)
            for i in pairs:
                q = q0 + i
                slot = q % 2
                while not PEMPTY[slot].done(((q // 2) & 1) ^ 1):
                    yield
                if form == "alternate_pairs":
                    mine = [j for j in (2 * i, 2 * i + 1) if j < nkb]
                elif form == "item_local":
                    mine = [j for j in (2 * i + r,) if j < nkb]
                else:
                    mine = [j for j in (2 * i, 2 * i + 1) if j < nkb and (kbase + j) % 2 == r]
                for j in mine:
                    jin = j % per_atom
                    first = (j == mine[0] or jin == 0) if form == "alternate_pairs" else (jin < 2 or per_atom == 1)
                    if first:
                        kt = kt_item + j // per_atom
                        while kt_cur < kt:
                            kt_cur, st = kt_cur + 1, st + 1
                            if st == stages:
                                st, ph = 0, ph ^ 1
                        while not FULL[st].done(ph):
                            yield
                    if stage_tag[st] != kt_item + j // per_atom:
                        raise Stale(f"issuer {r} read stage {st} holding k-tile {stage_tag[st]}")
                    buf_tag[2 * slot + (j - 2 * i)] = (q, j, kt_item)
                    last = (j == mine[-1] or jin == per_atom - 1) if form == "alternate_pairs" else \
                        (jin + 2 >= per_atom or j + 2 >= nkb)
                    if last:
                        pending.append((r, EMPTY[st]))
                pending.append((r, PFULL[slot]))
                yield
            q0 += npairs
            kt_item += kc
            kbase += nkb

    def epilogue():
        q, kt_item = 0, 0
        for kc in items:
            nkb = kc * per_atom
            for j in range(0, nkb, 2):
                slot = q % 2
                while not PFULL[slot].done((q // 2) & 1):
                    yield
                if buf_tag[2 * slot] != (q, j, kt_item) or (j + 1 < nkb and buf_tag[2 * slot + 1] != (q, j + 1, kt_item)):
                    raise Stale(f"epilogue read pair {q} from buffers holding {buf_tag[2 * slot:2 * slot + 2]}")
                PEMPTY[slot].arrive()
                q += 1
            kt_item += kc

    def complete_one():
        if pending:
            r = rng.choice([p[0] for p in pending])
            k = next(i for i, p in enumerate(pending) if p[0] == r)
            pending.pop(k)[1].arrive()

    agents = [producer(), issuer(0), issuer(1)] + [epilogue() for _ in range(8)]
    alive, idle = list(range(len(agents))), 0
    while alive:
        if rng.random() < 0.3:
            complete_one()
        a = rng.choice(alive)
        try:
            next(agents[a])
            idle += 1
        except StopIteration:
            alive.remove(a)
            idle = 0
        if idle > 50000:
            raise AssertionError(f"deadlock: agents {alive} still waiting")
    while pending:
        complete_one()


def _items(rng):
    return [rng.randint(1, 9) for _ in range(rng.randint(1, 6))]


@pytest.mark.parametrize("bk", [32, 64, 128])
@pytest.mark.parametrize("stages", [2, 3, 4, 6])
def test_protocol_completes_without_stale_reads(bk, stages):
    rng = random.Random(1000 * bk + stages)
    for trial in range(12):
        run(_items(rng), bk, stages, trial)
    # runs of one-k-block items (K <= 128 at 128-wide k-blocks) and odd item lengths
    for trial in range(6):
        run([1] * rng.randint(1, 10) + [rng.randint(1, 5)] + [1] * rng.randint(0, 6), bk, stages, 100 + trial)


def test_model_catches_the_earlier_forms_hazards():
    # alternate pairs: an issuer skips up to three k-tiles of the other, so on a two-stage ring
    # its first wait can match a stage's earlier phase
    with pytest.raises(Stale):
        for seed in range(20):
            run([3, 5, 2, 1, 2, 3, 4, 5], 128, 2, seed, form="alternate_pairs")
    # pair roles fixed by position inside the item: runs of one-k-block items give issuer 0
    # every k-block, so issuer 1's first wait lands any number of k-tiles later
    with pytest.raises(Stale):
        for seed in range(20):
            run([1, 2, 3, 4, 5], 128, 2, seed, form="item_local")
    # while the alternate-pairs form is sound on the four-stage rings it then required
    for seed in range(10):
        run([3, 5, 2, 1, 2, 3, 4, 5], 128, 4, seed, form="alternate_pairs")
