"""Host model of the dK/dV kernel's coordination protocol (no GPU).

Key tiles are handed out at run time through a 4-entry ring; per unit the
producer loads K and V, then per step Q_i (3-slot ring), dO_i (2-slot ring)
and the step's -LSE/-D vectors (2-slot ring, released by the warpgroups).
The issuer meets the relay warp at a named barrier (no time limit) before
each MMA group: per step S^T(s), dK(s-1) (dS^T(s-1) ready), dP^T(s) (dO_i
landed), dV(s) (P^T(s) handed over; at s = 0 also the previous unit's dK, dV
stored), and the unit's last dK.  At d = 64 tensor memory holds two S^T
buffers, so S^T(s+1) is issued after dP^T(s) and before dV(s); the P^T
hand-off barrier then alternates with the buffer as well, because the
warpgroups can hand P^T(s+1) over before the relay has waited for P^T(s)
(the model catches a single hand-off barrier in that order).

The model runs the roles as threads with the kernel's loop structure over a
mix of units (including one-step units), mbarriers as phase counters with
arrival counts (a waiter that sees a later phase of the same parity waits
for the next one, as on the GPU), waits that fail at random injected points,
and checks that a clean run stores every unit, that no injected failure
leaves a role blocked at a named barrier, and that the relay and the issuer
leave together at the unit after an abort.
"""
import random
import threading

import pytest

from test_fwd_protocol_model import Hang, MBar, Rendezvous

WAIT_LIMIT_S = 0.05
UNITS = [4, 1, 3, 2, 5, 1]  # steps of each unit
Q_SLOTS, DO_SLOTS, UNIT_SLOTS = 3, 2, 4


class CTA:
    def __init__(self, fail_p, seed, double_s, alt_p=True, jitter=0.0):
        self.rng = random.Random(seed)
        self.fail_p, self.double_s, self.alt_p, self.jitter = fail_p, double_s, alt_p, jitter
        self.lock = threading.Lock()
        self.abort = False
        self.kv_full, self.kv_empty = MBar(), MBar()
        self.q_full = [MBar() for _ in range(Q_SLOTS)]
        self.q_empty = [MBar() for _ in range(Q_SLOTS)]
        self.do_full = [MBar(2) for _ in range(DO_SLOTS)]  # TMA + the vector writer
        self.do_empty = [MBar() for _ in range(DO_SLOTS)]
        self.vec_empty = [MBar(2) for _ in range(DO_SLOTS)]
        self.s_full = [MBar(), MBar()]
        self.dp_full = MBar()
        self.p_ready = [MBar(2), MBar(2)]
        self.ds_ready = MBar(2)
        self.dkv_full, self.dkv_free = MBar(), MBar(2)
        self.unit_full = [MBar() for _ in range(UNIT_SLOTS)]
        self.unit_empty = [MBar(4) for _ in range(UNIT_SLOTS)]  # issuer, relay, 2 warpgroups
        self.ring = [None] * UNIT_SLOTS
        self.next_unit = 0
        self.rv = Rendezvous("kBarRelay")
        self.stored = 0

    def wait(self, bar, parity):
        with self.lock:
            if self.abort or self.rng.random() < self.fail_p:
                self.abort = True
                return False
        with bar.cv:
            bar.cv.wait_for(lambda: bar.done(parity) or self.abort, timeout=WAIT_LIMIT_S)
            if bar.done(parity):
                return True
        with self.lock:
            self.abort = True
        return False

    def pause(self):
        if self.jitter:
            with self.lock:
                d = self.rng.random() * self.jitter
            threading.Event().wait(d)

    def p_bar(self, st):
        if self.double_s and self.alt_p:
            return self.p_ready[st & 1], (st >> 1) & 1
        return self.p_ready[0], st & 1

    def s_bar(self, st):
        if self.double_s:
            return self.s_full[st & 1], (st >> 1) & 1
        return self.s_full[0], st & 1


def read(c, un):
    us = un % UNIT_SLOTS
    u = c.ring[us]
    c.unit_empty[us].arrive()
    return u


def producer(c):
    kv_it = st = un = 0
    while True:
        us = un % UNIT_SLOTS
        if not c.wait(c.unit_empty[us], ((un // UNIT_SLOTS) & 1) ^ 1):
            return
        u = c.next_unit if c.next_unit < len(UNITS) else -1
        c.next_unit += 1
        c.ring[us] = u
        c.unit_full[us].arrive()
        un += 1
        if u < 0:
            return
        if not c.wait(c.kv_empty, (kv_it & 1) ^ 1):
            return
        c.kv_full.arrive()
        kv_it += 1
        for _ in range(UNITS[u]):
            qs, ds = st % Q_SLOTS, st % DO_SLOTS
            if not c.wait(c.q_empty[qs], ((st // Q_SLOTS) & 1) ^ 1):
                return
            c.q_full[qs].arrive()
            if not c.wait(c.do_empty[ds], ((st // DO_SLOTS) & 1) ^ 1):
                return
            c.do_full[ds].arrive()                          # the tile's bytes
            if not c.wait(c.vec_empty[ds], ((st // DO_SLOTS) & 1) ^ 1):
                return
            c.do_full[ds].arrive()                          # the vectors
            st += 1


def issuer(c):
    st = un = 0
    aborted = False
    while True:
        aborted = c.rv.go(aborted)                          # unit published
        if aborted:
            return
        u = read(c, un)
        un += 1
        if u < 0:
            return
        n = UNITS[u]

        def issue_s(step):
            bar, _ = c.s_bar(step)
            bar.arrive()

        if c.double_s:
            aborted = c.rv.go(aborted)                      # S^T(0)
            if not aborted:
                issue_s(st)
        for s in range(n):
            ds = st % DO_SLOTS
            if not c.double_s:
                aborted = c.rv.go(aborted)                  # S^T(s)
                if not aborted:
                    issue_s(st)
            if s > 0:
                aborted = c.rv.go(aborted)                  # dK(s-1)
                if not aborted:
                    c.q_empty[(st - 1) % Q_SLOTS].arrive()
            aborted = c.rv.go(aborted)                      # dP^T(s)
            if not aborted:
                c.dp_full.arrive()
            if c.double_s and s + 1 < n:
                aborted = c.rv.go(aborted)                  # S^T(s+1)
                if not aborted:
                    issue_s(st + 1)
            aborted = c.rv.go(aborted)                      # dV(s)
            if not aborted:
                c.do_empty[ds].arrive()
            st += 1
        aborted = c.rv.go(aborted)                          # the unit's last dK
        if not aborted:
            c.q_empty[(st - 1) % Q_SLOTS].arrive()
            c.dkv_full.arrive()
            c.kv_empty.arrive()


def relay(c):
    kv_it = st = unit_it = un = 0
    aborted = False

    def wait(bar, parity):
        nonlocal aborted
        if not aborted:
            aborted = not c.wait(bar, parity)

    while True:
        wait(c.unit_full[un % UNIT_SLOTS], (un // UNIT_SLOTS) & 1)
        aborted = c.rv.go(aborted)
        if aborted:
            return
        u = read(c, un)
        un += 1
        if u < 0:
            return
        n = UNITS[u]
        wait(c.kv_full, kv_it & 1)
        kv_it += 1
        if c.double_s:
            wait(c.q_full[st % Q_SLOTS], (st // Q_SLOTS) & 1)
            aborted = c.rv.go(aborted)
        for s in range(n):
            if not c.double_s:
                wait(c.q_full[st % Q_SLOTS], (st // Q_SLOTS) & 1)
                aborted = c.rv.go(aborted)
            if s > 0:
                wait(c.ds_ready, (st - 1) & 1)
                aborted = c.rv.go(aborted)
            wait(c.do_full[st % DO_SLOTS], (st // DO_SLOTS) & 1)
            aborted = c.rv.go(aborted)
            if c.double_s and s + 1 < n:
                n1 = st + 1
                wait(c.q_full[n1 % Q_SLOTS], (n1 // Q_SLOTS) & 1)
                aborted = c.rv.go(aborted)
            if s == 0 and unit_it > 0:
                wait(c.dkv_free, (unit_it - 1) & 1)
            c.pause()  # a relay slowed down here must still see P^T(s)
            bar, par = c.p_bar(st)
            wait(bar, par)
            aborted = c.rv.go(aborted)
            st += 1
        wait(c.ds_ready, (st - 1) & 1)
        aborted = c.rv.go(aborted)
        unit_it += 1


def warpgroup(c):
    st = unit_it = un = 0
    while True:
        if not c.wait(c.unit_full[un % UNIT_SLOTS], (un // UNIT_SLOTS) & 1):
            return
        u = read(c, un)
        un += 1
        if u < 0:
            return
        for _ in range(UNITS[u]):
            sbar, spar = c.s_bar(st)
            if not c.wait(sbar, spar):
                return
            if not c.wait(c.do_full[st % DO_SLOTS], (st // DO_SLOTS) & 1):
                return
            bar, _ = c.p_bar(st)
            bar.arrive()
            if not c.wait(c.dp_full, st & 1):
                return
            c.ds_ready.arrive()
            c.vec_empty[st % DO_SLOTS].arrive()
            st += 1
        if not c.wait(c.dkv_full, unit_it & 1):
            return
        unit_it += 1
        with c.lock:
            c.stored += 1
        c.dkv_free.arrive()


def run(fail_p, seed, double_s, alt_p=True, jitter=0.0):
    c = CTA(fail_p, seed, double_s, alt_p, jitter)
    hangs = []

    def wrap(f):
        try:
            f(c)
        except Hang as e:
            hangs.append(str(e))

    roles = [producer, issuer, relay, warpgroup, warpgroup]
    threads = [threading.Thread(target=wrap, args=(f,), daemon=True) for f in roles]
    for th in threads:
        th.start()
    for th in threads:
        th.join(12.0)
    return c, hangs, sum(th.is_alive() for th in threads)


@pytest.mark.parametrize("double_s", [False, True])
def test_clean_schedule_stores_every_unit(double_s):
    c, hangs, alive = run(0.0, 0, double_s)
    assert not hangs and alive == 0 and not c.abort
    assert c.stored == 2 * len(UNITS)


@pytest.mark.parametrize("double_s", [False, True])
def test_slow_relay_still_sees_every_hand_off(double_s):
    # the relay pauses before each P^T wait, so the warpgroups run ahead
    c, hangs, alive = run(0.0, 1, double_s, jitter=0.01)
    assert not hangs and alive == 0 and not c.abort
    assert c.stored == 2 * len(UNITS)


def test_model_catches_a_single_hand_off_barrier_with_two_buffers():
    found = False
    for seed in range(6):
        c, hangs, alive = run(0.0, 10 + seed, True, alt_p=False, jitter=0.01)
        if hangs or alive or c.abort or c.stored < 2 * len(UNITS):
            found = True
            break
    assert found


@pytest.mark.parametrize("double_s", [False, True])
@pytest.mark.parametrize("seed", range(12))
def test_injected_wait_failures_never_hang(double_s, seed):
    fail_p = [0.005, 0.02, 0.1, 0.3][seed % 4]
    _, hangs, alive = run(fail_p, 100 + seed, double_s)
    assert not hangs and alive == 0, hangs
