"""Host model of the forward kernel's coordination protocol (no GPU).

The forward kernel's issuer meets the softmax warpgroups (P_t handed over)
and the relay warp (Q/K/V landed) at named barriers, which have no time
limit.  Its abort rule: after a bounded mbarrier wait runs out, no role leaves
early; every role walks its deterministic schedule to the end with waits and
work skipped, so every barrier generation still pairs up.  This file models
the five roles (producer, relay, issuer, softmax 0/1) as threads with the
kernel's loop structure over a mix of causal query-tile pairs, named barriers
as OR-reducing rendezvous and mbarriers as phase counters whose waits fail at
randomly injected points, and checks that
  * a clean run finishes every epilogue,
  * no injected failure leaves a role blocked at a rendezvous,
  * the model does catch the hang of a variant whose softmax leaves early.
"""
import random
import threading

import pytest

WAIT_LIMIT_S = 0.05   # bounded mbarrier wait of the model
HANG_S = 3.0          # a rendezvous not completed in this time is a hang
UNITS = [(7, 0), (5, 6), (3, 4), (1, 2), (4, 4)]  # (blocks of tile 0, tile 1)
SLOTS = 4


class Hang(Exception):
    pass


class Rendezvous:
    """Named barrier over two roles returning the OR of their predicates."""

    def __init__(self, name):
        self.name = name
        self.cv = threading.Condition()
        self.count, self.acc, self.gen, self.res = 0, False, 0, {}

    def go(self, pred):
        with self.cv:
            g = self.gen
            self.acc |= pred
            self.count += 1
            if self.count == 2:
                self.res[g], self.count, self.acc = self.acc, 0, False
                self.gen += 1
                self.cv.notify_all()
            elif not self.cv.wait_for(lambda: self.gen > g, timeout=HANG_S):
                raise Hang(f"{self.name} generation {g}")
            return self.res[g]


class MBar:
    """mbarrier: a phase completes after `count` arrivals."""

    def __init__(self, count=1):
        self.count, self.pending, self.phase = count, count, 0
        self.cv = threading.Condition()

    def arrive(self):
        with self.cv:
            self.pending -= 1
            if self.pending == 0:
                self.pending = self.count
                self.phase += 1
                self.cv.notify_all()

    def done(self, parity):
        return (self.phase & 1) != parity


class CTA:
    def __init__(self, fail_p, seed, softmax_leaves_early=False):
        self.rng = random.Random(seed)
        self.fail_p = fail_p
        self.early = softmax_leaves_early
        self.lock = threading.Lock()
        self.abort = False
        self.qfull, self.qempty = [MBar(), MBar()], [MBar(), MBar()]
        self.sfull, self.ofull = [MBar(), MBar()], [MBar(), MBar()]
        self.kvfull = [MBar() for _ in range(SLOTS)]
        self.kvempty = [MBar() for _ in range(SLOTS)]
        self.kv = Rendezvous("kBarKv")
        self.p = [Rendezvous("kBarP+0"), Rendezvous("kBarP+1")]
        self.epilogues = 0

    def wait(self, bar, parity):
        with self.lock:
            if self.rng.random() < self.fail_p:
                self.abort = True
                return False
        with bar.cv:
            bar.cv.wait_for(lambda: bar.done(parity) or self.abort, timeout=WAIT_LIMIT_S)
            if bar.done(parity):
                return True
        with self.lock:
            self.abort = True
        return False


def producer(c):
    kv_it, q_it = 0, [0, 0]
    for nb in UNITS:
        for t in range(2):
            if nb[t] == 0:
                continue
            if not c.wait(c.qempty[t], (q_it[t] & 1) ^ 1):
                return
            c.qfull[t].arrive()
            q_it[t] += 1
        for _ in range(max(nb)):
            for _ in range(2):  # K_j, V_j
                slot = kv_it % SLOTS
                if not c.wait(c.kvempty[slot], ((kv_it // SLOTS) & 1) ^ 1):
                    return
                c.kvfull[slot].arrive()
                kv_it += 1


def relay(c):
    kv_it, q_it, aborted = 0, [0, 0], False

    def kv_ready():
        nonlocal kv_it, aborted
        slot, par = kv_it % SLOTS, (kv_it // SLOTS) & 1
        kv_it += 1
        if not aborted:
            aborted = not c.wait(c.kvfull[slot], par)

    for nb in UNITS:
        nbmax = max(nb)
        for t in range(2):
            if nb[t] == 0:
                continue
            par = q_it[t] & 1
            q_it[t] += 1
            if not aborted:
                aborted = not c.wait(c.qfull[t], par)
        kv_ready()
        aborted = c.kv.go(aborted)
        for j in range(nbmax):
            kv_ready()
            if j + 1 < nbmax:
                kv_ready()
            aborted = c.kv.go(aborted)


def issuer(c):
    kv_it, aborted = 0, False
    for nb in UNITS:
        nbmax = max(nb)
        aborted = c.kv.go(aborted)
        kslot = kv_it % SLOTS
        kv_it += 1
        if not aborted:
            for t in range(2):
                if nb[t] > 0:
                    c.sfull[t].arrive()
                    if nb[t] == 1:
                        c.qempty[t].arrive()
            c.kvempty[kslot].arrive()
        for j in range(nbmax):
            aborted = c.kv.go(aborted)
            vslot = kv_it % SLOTS
            kv_it += 1
            have_next = j + 1 < nbmax
            if have_next:
                kslot = kv_it % SLOTS
                kv_it += 1
            for t in range(2):
                if j >= nb[t]:
                    continue
                aborted = c.p[t].go(aborted)
                if aborted:
                    continue
                if j == nb[t] - 1:
                    c.ofull[t].arrive()
                if j + 1 < nb[t]:
                    c.sfull[t].arrive()
                    if j + 1 == nb[t] - 1:
                        c.qempty[t].arrive()
            if not aborted:
                c.kvempty[vslot].arrive()
                if have_next:
                    c.kvempty[kslot].arrive()


def softmax(c, t):
    s_it = o_it = 0
    aborted = False
    for nb in UNITS:
        if nb[t] == 0:
            continue
        for _ in range(nb[t]):
            par = s_it & 1
            s_it += 1
            if not aborted:
                aborted = not c.wait(c.sfull[t], par)
            if aborted and c.early:
                return
            aborted = c.p[t].go(aborted)
        par = o_it & 1
        o_it += 1
        if not aborted:
            aborted = not c.wait(c.ofull[t], par)
        if not aborted:
            with c.lock:
                c.epilogues += 1


def run(fail_p, seed, softmax_leaves_early=False):
    c = CTA(fail_p, seed, softmax_leaves_early)
    hangs = []

    def wrap(f, *a):
        try:
            f(c, *a)
        except Hang as e:
            hangs.append(str(e))

    roles = [(producer, ()), (relay, ()), (issuer, ()), (softmax, (0,)), (softmax, (1,))]
    threads = [threading.Thread(target=wrap, args=(f,) + a, daemon=True) for f, a in roles]
    for th in threads:
        th.start()
    for th in threads:
        th.join(4 * HANG_S)
    alive = sum(th.is_alive() for th in threads)
    return c, hangs, alive


def test_clean_schedule_finishes_every_epilogue():
    c, hangs, alive = run(0.0, 0)
    assert not hangs and alive == 0
    assert c.epilogues == sum(1 for nb in UNITS for t in range(2) if nb[t] > 0)


@pytest.mark.parametrize("seed", range(24))
def test_injected_wait_failures_never_hang(seed):
    fail_p = [0.005, 0.02, 0.1, 0.3][seed % 4]
    _, hangs, alive = run(fail_p, seed)
    assert not hangs and alive == 0, hangs


def test_model_catches_softmax_that_leaves_early():
    found = False
    for seed in range(6):
        _, hangs, alive = run(0.3, 100 + seed, softmax_leaves_early=True)
        if hangs or alive:
            found = True
            break
    assert found
