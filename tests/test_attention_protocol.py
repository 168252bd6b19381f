"""A model of the attention kernel's synchronisation protocol, run on the CPU.

The tcgen05 attention kernel has four roles per CTA: a TMA producer (Q once,
then K and V tiles through two 2-stage rings), one MMA-issuing thread, and two
softmax warpgroups (query tiles A and B).  They synchronise only through
mbarriers, and the tensor core runs MMAs and commits in issue order.  This
model replays those roles as coroutines under random interleavings, with
mbarrier semantics (arrival counts, transaction bytes, phase parity: a wait
on parity P passes once the phase with that parity has completed) and an
in-order tensor pipe, and checks that

* every interleaving finishes (no role waits forever), and
* every MMA reads what it should: S(j) the Q tile and the K tile j, PV(j) the
  V tile j and the P of tile j (written by the softmax, not yet overwritten
  by the next S), the softmax the scores of tile j, the output step O after
  the last PV.

The roles issue exactly the waits, arrivals and commits of the kernel, in its
order (issue order per key tile j: S_A(j), PV_B(j-1), S_B(j), PV_A(j)).
Planted mistakes in the model (a K stage released before S_B read it, S_B
issued before PV_B(j-1), an arrival before P is written) must be caught.
"""

import random

import pytest


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.tx, self.completed = name, count, count, 0, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, f"{self.name}: more arrivals than its count"
        self._complete()

    def expect_tx(self, n):
        self.tx += n

    def tx_done(self, n):
        self.tx -= n
        self._complete()

    def _complete(self):
        if self.pending == 0 and self.tx == 0:
            self.completed += 1
            self.pending = self.count

    def passed(self, parity):
        # the phase with this parity has completed (a fresh barrier passes parity 1)
        return (self.completed & 1) != parity


class Kernel:
    """One CTA over nt key tiles.  `plant` names a deliberate mistake."""

    def __init__(self, nt, seed, plant=None):
        self.nt, self.rng, self.plant = nt, random.Random(seed), plant
        B = Barrier
        self.q_full = B("q_full", 1)
        self.k_full = [B(f"k_full{s}", 1) for s in range(2)]
        self.k_empty = [B(f"k_empty{s}", 1) for s in range(2)]
        self.v_full = [B(f"v_full{s}", 1) for s in range(2)]
        self.v_empty = [B(f"v_empty{s}", 1) for s in range(2)]
        self.s_full = [B(f"s_full{x}", 1) for x in range(2)]
        self.p_full = [B(f"p_full{x}", 1) for x in range(2)]    # one arrival per softmax group here
        self.o_done = [B(f"o_done{x}", 1) for x in range(2)]
        self.drain = B("drain", 1)
        self.pipe, self.copies = [], []
        self.q_loaded = False
        self.k_stage, self.v_stage = [None, None], [None, None]
        self.tmem_s = [None, None]                                # ("S", j) scores or ("P", j) probabilities
        self.pv_done = [set(), set()]
        self.finished = set()

    @staticmethod
    def wait(bar, parity):
        while not bar.passed(parity):
            yield (bar, parity)

    # ------------------------------------------------------------- roles
    def producer(self):
        self.q_full.expect_tx(1)
        self.q_full.arrive()
        self.copies.append((self.q_full, "Q", 0, 0))

        def load(is_k, j):
            s, ph = j % 2, (j // 2) & 1
            yield from self.wait((self.k_empty if is_k else self.v_empty)[s], ph ^ 1)
            full = (self.k_full if is_k else self.v_full)[s]
            full.expect_tx(1)
            full.arrive()
            self.copies.append((full, "K" if is_k else "V", s, j))

        yield from load(True, 0)
        for j in range(self.nt):
            if j + 1 < self.nt:
                yield from load(True, j + 1)
            yield from load(False, j)
        yield from self.wait(self.q_full, 0)

    def issuer(self):
        nt = self.nt

        def pv(x, j):
            yield from self.wait(self.p_full[x], j & 1)
            self.pipe += [("PV", x, j % 2, j), ("commit", self.o_done[x])]

        yield from self.wait(self.q_full, 0)
        for j in range(nt):
            s, ph = j % 2, (j // 2) & 1
            yield from self.wait(self.k_full[s], ph)
            self.pipe += [("S", 0, s, j), ("commit", self.s_full[0])]
            if self.plant == "k_released_early":
                self.pipe.append(("commit", self.k_empty[s]))
            if self.plant == "s_b_before_pv_b":
                self.pipe += [("S", 1, s, j), ("commit", self.s_full[1])]
            if j >= 1:
                yield from pv(1, j - 1)
                self.pipe.append(("commit", self.v_empty[(j - 1) % 2]))
            if self.plant != "s_b_before_pv_b":
                self.pipe += [("S", 1, s, j), ("commit", self.s_full[1])]
            if self.plant != "k_released_early":
                self.pipe.append(("commit", self.k_empty[s]))
            yield from self.wait(self.v_full[s], ph)
            yield from pv(0, j)
        yield from pv(1, nt - 1)
        self.pipe.append(("commit", self.v_empty[(nt - 1) % 2]))
        self.pipe.append(("commit", self.drain))
        yield from self.wait(self.drain, 0)

    def softmax(self, x):
        for j in range(self.nt):
            yield from self.wait(self.s_full[x], j & 1)
            if j > 0:
                yield from self.wait(self.o_done[x], (j - 1) & 1)
                assert (j - 1) in self.pv_done[x], "O rescaled before PV(j-1) finished"
            assert self.tmem_s[x] == ("S", j), f"softmax {x} tile {j} read {self.tmem_s[x]}"
            if self.plant == "arrive_before_p":
                self.p_full[x].arrive()
                yield None
                self.tmem_s[x] = ("P", j)
            else:
                yield None                      # the exponentials
                self.tmem_s[x] = ("P", j)
                self.p_full[x].arrive()
            yield None
        yield from self.wait(self.o_done[x], (self.nt - 1) & 1)
        assert self.pv_done[x] == set(range(self.nt)), "output read before the last PV"

    # ------------------------------------------------------------- engines
    def tensor_step(self):
        op = self.pipe.pop(0)
        if op[0] == "commit":
            op[1].arrive()
        elif op[0] == "S":
            _, x, s, j = op
            assert self.q_loaded and self.k_stage[s] == j, f"S{x}({j}) read K stage {s} = {self.k_stage[s]}"
            cur = self.tmem_s[x]
            assert cur is None or (cur[0] == "P" and cur[1] in self.pv_done[x]), f"S{x}({j}) overwrote {cur}"
            self.tmem_s[x] = ("S", j)
        else:
            _, x, s, j = op
            assert self.v_stage[s] == j, f"PV{x}({j}) read V stage {s} = {self.v_stage[s]}"
            assert self.tmem_s[x] == ("P", j), f"PV{x}({j}) read {self.tmem_s[x]}"
            self.pv_done[x].add(j)

    def copy_step(self, i):
        bar, kind, s, j = self.copies.pop(i)
        if kind == "Q":
            self.q_loaded = True
        elif kind == "K":
            self.k_stage[s] = j
        else:
            self.v_stage[s] = j
        bar.tx_done(1)

    def run(self):
        roles = {"tma": self.producer(), "mma": self.issuer(), "A": self.softmax(0), "B": self.softmax(1)}
        blocked = {}
        for _ in range(200_000):
            choices = [("role", r) for r in roles
                       if r not in self.finished and (r not in blocked or blocked[r][0].passed(blocked[r][1]))]
            if self.pipe:
                choices.append(("pipe", None))
            choices += [("copy", i) for i in range(len(self.copies))]
            if not choices:
                assert len(self.finished) == 4, "deadlock: " + ", ".join(
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


@pytest.mark.parametrize("nt", [1, 2, 3, 4, 7])
def test_protocol_finishes_and_reads_the_right_buffers(nt):
    for seed in range(60):
        Kernel(nt, seed * 977 + nt).run()


@pytest.mark.parametrize("plant", ["k_released_early", "s_b_before_pv_b", "arrive_before_p"])
def test_planted_mistakes_are_caught(plant):
    caught = 0
    for nt in (2, 3, 5):
        for seed in range(40):
            try:
                Kernel(nt, seed, plant).run()
            except AssertionError:
                caught += 1
    assert caught > 0, f"the model missed the planted mistake {plant}"
