"""A model of the tcgen05 attention kernel's synchronisation protocol (not the kernel
itself), explored over random schedules on the CPU.

Three roles share a CTA: the producers (one actor standing for all 256 threads), the
MMA issuer and the softmax (one actor for its 128 rows).  They meet on mbarriers whose
waits test a phase parity: ``try_wait.parity(p)`` succeeds when the barrier's current
phase has the other parity, so a waiter that is two phases behind what it means to wait
for sees its phase as complete.  The asynchronous MMAs complete in issue order only
among MMAs into the same accumulator; a commit arrives once every MMA issued before it
has completed.

The model replays the kernel's waits, arrivals and commits as they are written, and
checks on every schedule that:
- every parity wait means the phase it returns for (no wait two phases behind);
- every buffer holds the tile its reader expects for the whole read: K_hat and the two
  V_hat stages (producers -> MMAs), the two S column sets of TMEM (S from Q K^T, then
  the softmax's P over it, read by P V), O (the P V sums, read at the end), and the
  4-slot rings of per-tile data the softmax reads;
- every schedule ends with every role done.
No property rests on timing: the schedules are arbitrary interleavings.  Three earlier
versions of the protocol are kept as switches, and the model must find their races:
Q K^T of tile j issued once P V of tile j - 2 was issued (not completed); the epilogue
waiting on the per-P V barrier with the last tile's parity; and the producers publishing
tile j's keys without waiting for the softmax's P_FULL of tile j - 2, where the
softmax's K_FULL wait for tile j - 2 can then find the barrier two phases ahead (the
kernel once relied on the softmax being fast enough instead).
"""

import random

import pytest


class Bar:
    def __init__(self, name):
        self.name, self.done = name, 0        # completed phases

    def test(self, phase, log):
        """try_wait.parity for `phase`; records a wait whose answer is not about `phase`."""
        ok = (self.done & 1) != (phase & 1)
        if ok != (self.done > phase):
            log.append(f"{self.name}: waiting for phase {phase} with {self.done} complete")
        return ok


class Model:
    def __init__(self, T, seed, old_qk_rule=False, old_epilogue=False, old_publish=False, kbuf=1, old_kbuf_wait=False):
        self.T, self.rng = T, random.Random(seed)
        self.kbuf = kbuf                      # K_hat buffers (2 in the CTA-pair kernel)
        self.old_kbuf_wait = old_kbuf_wait    # with 2 buffers, wait only for Q K^T of tile j - 1 to start
        self.old_qk_rule, self.old_epilogue = old_qk_rule, old_epilogue
        self.old_publish = old_publish
        names = ["K_FULL0", "K_FULL1", "V_FULL0", "V_FULL1", "V_EMPTY0", "V_EMPTY1", "S_FULL0", "S_FULL1",
                 "P_FULL0", "P_FULL1", "O_DONE", "K_EMPTY", "K_EMPTY0", "K_EMPTY1", "MMA_DONE"]
        self.bar = {n: Bar(n) for n in names}
        self.errors = []
        # buffer contents: what each holds now
        self.khat = [None, None]              # K_hat buffer b holds tile ...
        self.vhat = [None, None]
        self.s = [None, None]                 # ("S", j) after Q K^T, ("P", j) after the softmax
        self.o = set()                        # tiles whose P V is summed into O
        self.ring = [None] * 4                # per-tile data the softmax reads (lengths, steps)
        self.ops = []                         # issued, not completed MMAs: dicts
        self.commits = []                     # (barrier, ids of the MMAs it waits for)
        self.next_id = 0

    # ---- asynchronous MMAs -------------------------------------------------------
    def issue(self, kind, j):
        acc = ("S", j & 1) if kind == "QK" else ("O",)
        op = dict(id=self.next_id, kind=kind, j=j, acc=acc)
        self.next_id += 1
        # reads checked now and at completion: the operand must hold tile j throughout
        self.check_reads(op)
        self.ops.append(op)
        return op

    def check_reads(self, op):
        j = op["j"]
        if op["kind"] == "QK" and self.khat[j % self.kbuf] != j:
            self.errors.append(f"QK({j}) reads K_hat holding {self.khat[j % self.kbuf]}")
        if op["kind"] == "PV":
            if self.s[j & 1] != ("P", j):
                self.errors.append(f"PV({j}) reads P from S columns holding {self.s[j & 1]}")
            if self.vhat[j & 1] != j:
                self.errors.append(f"PV({j}) reads V_hat stage holding {self.vhat[j & 1]}")

    def commit(self, name):
        ids = {o["id"] for o in self.ops}
        if ids:
            self.commits.append((name, ids))
        else:
            self.bar[name].done += 1          # nothing in flight: arrives at once

    def completable(self):
        """MMAs that may complete now: the oldest pending one of each accumulator."""
        firsts = {}
        for o in self.ops:
            firsts.setdefault(o["acc"], o)
        return list(firsts.values())

    def complete(self, op):
        self.check_reads(op)
        self.ops.remove(op)
        j = op["j"]
        if op["kind"] == "QK":
            self.s[j & 1] = ("S", j)
        else:
            self.o.add(j)
        pending = {o["id"] for o in self.ops}
        still = []
        for name, ids in self.commits:
            if ids & pending:
                still.append((name, ids))
            else:
                self.bar[name].done += 1
        self.commits = still

    # ---- roles (generators: yield = give up the turn) --------------------------------
    def wait(self, name, phase):
        while not self.bar[name].test(phase, self.errors):
            yield

    def producers(self):
        for j in range(self.T):
            s = j & 1
            # the K_hat buffer of tile j is free once Q K^T of tile j - kbuf completed: one
            # barrier with one buffer; with two, each buffer's own barrier (one barrier for
            # both cannot express "tile j - 2" once tile j - 1 has also completed)
            if j >= self.kbuf:
                if self.kbuf == 1:
                    yield from self.wait("K_EMPTY", j - 1)
                elif self.old_kbuf_wait:
                    yield from self.wait("K_EMPTY", j - 2)
                else:
                    yield from self.wait(f"K_EMPTY{j & 1}", (j - 2) >> 1)
            self.khat[j % self.kbuf] = j
            self.ring[j & 3] = j
            # tile j is published only after the softmax finished tile j - 2
            if j >= 2 and not self.old_publish:
                yield from self.wait(f"P_FULL{s}", (j - 2) >> 1)
            self.bar[f"K_FULL{s}"].done += 1
            yield
            if j >= 2:
                yield from self.wait(f"V_EMPTY{s}", (j - 2) >> 1)
            self.vhat[s] = j
            self.bar[f"V_FULL{s}"].done += 1
            yield

    def mma(self):
        T, nq, np_ = self.T, 0, 0
        while np_ < T:
            if (np_ < nq and self.bar[f"P_FULL{np_ & 1}"].test(np_ >> 1, self.errors)
                    and self.bar[f"V_FULL{np_ & 1}"].test(np_ >> 1, self.errors)):
                self.issue("PV", np_)
                self.commit("O_DONE")
                self.commit(f"V_EMPTY{np_ & 1}")
                np_ += 1
            elif (nq < T and nq <= np_ + 1 and self.bar[f"K_FULL{nq & 1}"].test(nq >> 1, self.errors)
                  and (nq < 2 or self.old_qk_rule
                       or self.bar[f"V_EMPTY{nq & 1}"].test((nq - 2) >> 1, self.errors))):
                self.issue("QK", nq)
                self.commit(f"S_FULL{nq & 1}")
                self.commit("K_EMPTY" if self.kbuf == 1 or self.old_kbuf_wait else f"K_EMPTY{nq & 1}")
                nq += 1
            yield
        self.commit("MMA_DONE")
        yield from self.wait("MMA_DONE", 0)

    def softmax(self):
        T = self.T
        for j in range(T):
            s = j & 1
            yield from self.wait(f"K_FULL{s}", j >> 1)
            if self.ring[j & 3] != j:
                self.errors.append(f"softmax({j}) reads ring slot holding {self.ring[j & 3]}")
            yield from self.wait(f"S_FULL{s}", j >> 1)
            if self.s[s] != ("S", j):
                self.errors.append(f"softmax({j}) reads S columns holding {self.s[s]}")
            if self.ring[j & 3] != j:
                self.errors.append(f"softmax({j}) reads ring slot holding {self.ring[j & 3]} after S")
            if j > 0 and self.rng.random() < 0.5:        # the running max grew: rescale O
                yield from self.wait("O_DONE", j - 1)
                if self.o != set(range(j)) or any(o["acc"] == ("O",) for o in self.ops):
                    self.errors.append(f"softmax({j}) rescales O holding {sorted(self.o)}")
            yield
            self.s[s] = ("P", j)
            self.bar[f"P_FULL{s}"].done += 1
            yield
        if T > 0:
            if self.old_epilogue:
                yield from self.wait("O_DONE", T - 1)
            else:
                yield from self.wait("MMA_DONE", 0)
            if self.o != set(range(T)):
                self.errors.append(f"epilogue reads O holding {sorted(self.o)} of {T} tiles")

    def run(self, max_steps=20000):
        roles = {"producers": self.producers(), "mma": self.mma(), "softmax": self.softmax()}
        for _ in range(max_steps):
            choices = list(roles) + ["async"] * (1 + len(self.ops))
            c = self.rng.choice(choices)
            if c == "async":
                ops = self.completable()
                if ops:
                    self.complete(self.rng.choice(ops))
                continue
            try:
                next(roles[c])
            except StopIteration:
                del roles[c]
            if not roles and not self.ops:
                return True
        self.errors.append("no progress: " + ", ".join(roles) + f" still running, {len(self.ops)} MMAs pending")
        return False


@pytest.mark.parametrize("T", [1, 2, 3, 5, 8])
def test_protocol_has_no_race(T):
    for seed in range(400):
        m = Model(T, seed)
        m.run()
        assert not m.errors, f"T={T} seed={seed}: {m.errors[:3]}"


def test_model_finds_the_qk_before_pv_race():
    """Q K^T of tile j once P V of tile j - 2 was only issued: a schedule exists where Q K^T
    completes first and overwrites the P that P V still reads."""
    hits = 0
    for seed in range(2000):
        m = Model(4, seed, old_qk_rule=True)
        m.run()
        hits += any("reads P from S columns" in e for e in m.errors)
    assert hits > 0


def test_model_finds_the_epilogue_parity_race():
    """The epilogue waiting on the per-P V barrier with the last tile's parity: a schedule
    exists where the barrier is two phases behind and the epilogue reads O early."""
    hits = 0
    for seed in range(2000):
        m = Model(2, seed, old_epilogue=True)
        m.run()
        hits += any("O_DONE: waiting for phase" in e or "epilogue reads O" in e for e in m.errors)
    assert hits > 0


def test_model_finds_the_unguarded_publish():
    """Without the P_FULL wait the producers can publish tile j + 2 before the softmax waits
    for tile j, and that wait is two phases behind."""
    hits = 0
    for seed in range(400):
        m = Model(3, seed, old_publish=True)
        m.run()
        hits += any(e.startswith("K_FULL") for e in m.errors)
    assert hits > 0


@pytest.mark.parametrize("T", [2, 3, 5, 8])
def test_two_key_buffers_have_no_race(T):
    """The CTA-pair kernel's two K_hat buffers: tile j is expanded into buffer j & 1 once Q K^T of
    tile j - 2 has completed (that buffer's own K_EMPTY barrier); on every schedule no wait is
    two phases off and every Q K^T reads its own tile."""
    for seed in range(400):
        m = Model(T, seed, kbuf=2)
        m.run()
        assert not m.errors, f"T={T} seed={seed}: {m.errors[:3]}"


def test_model_finds_the_shared_empty_barrier_race():
    """Two buffers behind one K_EMPTY barrier: waiting there for Q K^T of tile j - 2 fails once
    Q K^T of tile j - 1 has completed too (two phases past: the wait blocks)."""
    hits = 0
    for seed in range(2000):
        m = Model(6, seed, kbuf=2, old_kbuf_wait=True)
        m.run()
        hits += any(e.startswith("K_EMPTY") or "reads K_hat" in e for e in m.errors)
    assert hits > 0
