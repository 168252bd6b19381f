"""A model of the tcgen05 GEMM's synchronisation protocol, run on the CPU.

The persistent GEMM has three roles per CTA pair: a TMA producer filling a
6-stage operand ring (full / empty barriers), one MMA-issuing thread that
accumulates each tile into one of two TMEM accumulators (acc = local tile
index & 1) and commits the stage back and, after the tile's last k-block,
the accumulator to the epilogue (tmem_full), and the epilogue warps, which
drain an accumulator and hand it back (tmem_empty).  The roles are replayed
as coroutines under random interleavings with mbarrier semantics (counts,
transaction bytes, phase parity) and an in-order tensor pipe.  The model
checks that every interleaving finishes, that each MMA reads the stage
holding its (tile, k-block), that an accumulator is not restarted before the
epilogue has drained its previous tile, and that the epilogue reads complete
sums.  Each stage is filled by two copies (the B and the A operand).  The
one-CTA form runs a 4-stage ring and issues the B copies of its first stages
before it may read A (before the programmatic-dependent wait); the loop then
adds only their A copies.  With NVFP4 (fp8r) weights the one-CTA form keeps
three rings: A (five (four) stages), the codes (five (four), fed by a second
producer thread) and the expanded B stages (two); the epilogue warps expand each
k-block's codes into a B stage (after the MMAs have released it) before they
drain the unit's accumulator.  Planted mistakes (a stage released before its
MMAs, a wrong accumulator phase, more early stages than the ring holds, a B
stage rewritten without waiting for its MMAs) must be caught.
"""

import random

import pytest

from test_attention_protocol import Barrier


class Gemm:
    def __init__(self, tiles, num_kb, seed, plant=None, stages=6, pre=False, fp4=False, cstages=5):
        self.tiles, self.num_kb, self.plant, self.stages, self.pre = tiles, num_kb, plant, stages, pre
        self.fp4 = fp4                                   # codes expanded by the epilogue (NVFP4 or fp8r)
        self.bstages, self.cstages = (2, cstages) if fp4 else (stages, 0)
        self.cfull = [Barrier(f"cfull{s}", 1) for s in range(self.cstages)]
        self.cempty = [Barrier(f"cempty{s}", 1) for s in range(self.cstages)]
        self.bready = [Barrier(f"bready{s}", 1) for s in range(self.bstages)]
        self.bempty = [Barrier(f"bempty{s}", 1) for s in range(self.bstages)]
        self.code_holds = [None] * self.cstages
        self.rng = random.Random(seed)
        self.full = [Barrier(f"full{s}", 1) for s in range(stages)]
        self.empty = [Barrier(f"empty{s}", 1) for s in range(stages)]
        self.tmem_full = [Barrier(f"tmem_full{a}", 1) for a in range(2)]
        self.tmem_empty = [Barrier(f"tmem_empty{a}", 1) for a in range(2)]   # the epilogue's arrivals, as one
        self.drain = Barrier("drain", 1)
        self.pipe, self.copies = [], []
        self.stage_holds = [{} for _ in range(stages)]   # operand -> (tile, k-block)
        self.b_ring = [None] * self.bstages              # expanded B stages (NVFP4)
        self.acc = [None, None]            # (tile, k-blocks accumulated)
        self.drained = [set(), set()]      # tiles whose accumulator the epilogue has read out
        self.finished = set()

    @staticmethod
    def wait(bar, parity):
        while not bar.passed(parity):
            yield (bar, parity)

    def code_producer(self):
        n_pre = min(self.cstages, self.num_kb)          # before the programmatic wait
        for i in range(n_pre):
            self.cfull[i].expect_tx(1)
            self.cfull[i].arrive()
            self.copies.append((i, "C", (self.tiles[0], i)))
            yield None
        cs = cphase = it = 0
        for t in self.tiles:
            for kb in range(self.num_kb):
                if it >= n_pre:
                    yield from self.wait(self.cempty[cs], cphase ^ 1)
                    self.cfull[cs].expect_tx(1)
                    self.cfull[cs].arrive()
                    self.copies.append((cs, "C", (t, kb)))
                it += 1
                cs += 1
                if cs == self.cstages:
                    cs, cphase = 0, cphase ^ 1

    def producer(self):
        if self.fp4:                                    # A only: B comes from the expansion
            stage = phase = 0
            for t in self.tiles:
                for kb in range(self.num_kb):
                    yield from self.wait(self.empty[stage], phase ^ 1)
                    self.full[stage].expect_tx(1)
                    self.full[stage].arrive()
                    self.copies.append((stage, "A", (t, kb)))
                    stage += 1
                    if stage == self.stages:
                        stage, phase = 0, phase ^ 1
            return
        n_pre = min(self.stages, self.num_kb) if self.pre else 0
        if self.plant == "pre_overrun":
            n_pre = min(self.stages + 1, self.num_kb)
        for i in range(n_pre):                 # B halves of the first stages, before A may be read
            s = i % self.stages
            self.full[s].expect_tx(2)
            self.full[s].arrive()
            self.copies.append((s, "B", (self.tiles[0], i)))
            yield None
        stage = phase = it = 0
        for t in self.tiles:
            for kb in range(self.num_kb):
                if it >= n_pre:
                    yield from self.wait(self.empty[stage], phase ^ 1)
                    self.full[stage].expect_tx(2)
                    self.full[stage].arrive()
                    self.copies.append((stage, "B", (t, kb)))
                self.copies.append((stage, "A", (t, kb)))
                it += 1
                stage += 1
                if stage == self.stages:
                    stage, phase = 0, phase ^ 1

    def issuer(self):
        stage = phase = bstage = bphase = 0
        for local, t in enumerate(self.tiles):
            a = local & 1
            acc_phase = (local >> 1) & 1
            if self.plant == "wrong_acc_phase":
                acc_phase ^= 1
            yield from self.wait(self.tmem_empty[a], acc_phase ^ 1)
            for kb in range(self.num_kb):
                yield from self.wait(self.full[stage], phase)
                if self.fp4:
                    yield from self.wait(self.bready[bstage], bphase)
                if self.plant == "stage_released_early":
                    self.pipe.append(("commit", self.empty[stage]))
                self.pipe.append(("mma", a, stage, bstage, (t, kb)))
                if self.plant != "stage_released_early":
                    self.pipe.append(("commit", self.empty[stage]))
                if self.fp4:
                    self.pipe.append(("commit", self.bempty[bstage]))
                stage += 1
                if stage == self.stages:
                    stage, phase = 0, phase ^ 1
                bstage += 1
                if bstage == self.bstages:
                    bstage, bphase = 0, bphase ^ 1
            self.pipe.append(("commit", self.tmem_full[a]))
        self.pipe.append(("commit", self.drain))
        yield from self.wait(self.drain, 0)

    def epilogue(self):
        cs = cphase = bstage = bphase = 0
        for local, t in enumerate(self.tiles):
            a = local & 1
            if self.fp4:                                # expand the unit's k-blocks first
                for kb in range(self.num_kb):
                    yield from self.wait(self.cfull[cs], cphase)
                    if self.plant != "b_rewritten_early":
                        yield from self.wait(self.bempty[bstage], bphase ^ 1)
                    assert self.code_holds[cs] == (t, kb), f"expansion of ({t}, {kb}) read codes {self.code_holds[cs]}"
                    self.b_ring[bstage] = (t, kb)
                    self.bready[bstage].arrive()
                    self.cempty[cs].arrive()
                    yield None
                    cs += 1
                    if cs == self.cstages:
                        cs, cphase = 0, cphase ^ 1
                    bstage += 1
                    if bstage == self.bstages:
                        bstage, bphase = 0, bphase ^ 1
            yield from self.wait(self.tmem_full[a], (local >> 1) & 1)
            assert self.acc[a] == (t, self.num_kb), f"epilogue of tile {t} read {self.acc[a]}"
            yield None                       # reading the accumulator out
            self.drained[a].add(t)
            self.tmem_empty[a].arrive()

    def tensor_step(self):
        op = self.pipe.pop(0)
        if op[0] == "commit":
            op[1].arrive()
            return
        _, a, stage, bstage, (t, kb) = op
        held = self.stage_holds[stage]
        b = self.b_ring[bstage] if self.fp4 else held.get("B")
        assert held.get("A") == (t, kb) and b == (t, kb), f"MMA ({t}, {kb}) read stage {stage} = {held}, B {b}"
        if kb == 0:
            prev = self.acc[a]
            assert prev is None or prev[0] in self.drained[a], f"tile {t} restarted accumulator {a} over {prev}"
            self.acc[a] = (t, 1)
        else:
            assert self.acc[a] == (t, kb), f"accumulator {a} holds {self.acc[a]}, MMA ({t}, {kb})"
            self.acc[a] = (t, kb + 1)

    def copy_step(self, i):
        stage, operand, tag = self.copies.pop(i)
        if operand == "C":
            self.code_holds[stage] = tag
            self.cfull[stage].tx_done(1)
            return
        self.stage_holds[stage][operand] = tag
        self.full[stage].tx_done(1)

    def run(self):
        roles = {"tma": self.producer(), "mma": self.issuer(), "epi": self.epilogue()}
        if self.fp4:
            roles["codes"] = self.code_producer()
        blocked = {}
        for _ in range(400_000):
            choices = [("role", r) for r in roles
                       if r not in self.finished and (r not in blocked or blocked[r][0].passed(blocked[r][1]))]
            if self.pipe:
                choices.append(("pipe", None))
            choices += [("copy", i) for i in range(len(self.copies))]
            if not choices:
                assert len(self.finished) == len(roles), "deadlock: " + ", ".join(
                    f"{r} on {b.name}/{p}" for r, (b, p) in blocked.items())
                return
            kind, arg = self.rng.choice(choices)
            if kind == "pipe":
                self.tensor_step()
            elif kind == "copy":
                self.copy_step(arg)
            else:
                try:
                    y = next(roles[arg])
                    if y is None:
                        blocked.pop(arg, None)
                    else:
                        blocked[arg] = y
                except StopIteration:
                    self.finished.add(arg)
                    blocked.pop(arg, None)
        raise AssertionError("step limit")


FORMS = {"pair": dict(stages=6, pre=False), "one_cta": dict(stages=4, pre=True),
         "one_cta_nvfp4": dict(stages=5, fp4=True), "one_cta_fp8r": dict(stages=4, fp4=True, cstages=4)}


@pytest.mark.parametrize("form", sorted(FORMS))
@pytest.mark.parametrize("n_tiles,num_kb", [(1, 1), (1, 3), (1, 7), (2, 3), (3, 5), (5, 2), (6, 13)])
def test_protocol_finishes_and_reads_the_right_stages(form, n_tiles, num_kb):
    for seed in range(40):
        Gemm(list(range(10, 10 + n_tiles)), num_kb, seed * 31 + n_tiles, **FORMS[form]).run()


@pytest.mark.parametrize("form,plant", [("pair", "stage_released_early"), ("pair", "wrong_acc_phase"),
                                        ("one_cta", "stage_released_early"), ("one_cta", "pre_overrun"),
                                        ("one_cta_nvfp4", "stage_released_early"),
                                        ("one_cta_nvfp4", "b_rewritten_early"), ("one_cta_fp8r", "b_rewritten_early")])
def test_planted_mistakes_are_caught(form, plant):
    caught = 0
    for n_tiles, num_kb in ((3, 4), (4, 7), (2, 9)):
        for seed in range(40):
            try:
                Gemm(list(range(n_tiles)), num_kb, seed, plant, **FORMS[form]).run()
            except AssertionError:
                caught += 1
    assert caught > 0, f"the model missed the planted mistake {plant}"
