"""Host model of the dQ kernel's coordination protocol (no GPU).

Query tiles are handed out at run time: the producer takes the next one
from a counter and publishes it in a ring of 4 entries (-1 after the last),
which the relay (after waiting for the entry), the issuer (after meeting the
relay at its named barrier, U), and the warpgroups read and release.  The
issuer meets the relay warp at a named barrier (no time limit) before each
MMA group: per tile U, then per step j of a query tile, A (K_j, and at
j = 0 Q / dO, have landed), B for j > 0 (dS_{j-1} is ready; at j = 1 also the previous
tile's dQ has been stored), C (V_j has landed and S_j has been read); per
tile D (the last dS is ready).  The relay waits on the pipeline's mbarriers
(bounded); after a wait runs out both warps still walk the rest of the
tile's schedule with the abort bit carried by the barrier and leave together
at the next U, so every rendezvous pairs up.
The warpgroups and the producer use bounded mbarrier waits only and leave at
their first failed wait.

The model runs the five roles as threads with the kernel's loop structure
over a mix of tiles (including one-step tiles), mbarriers as phase counters
with arrival counts, waits that fail at random injected points, and checks
that
  * a clean run stores the dQ of every tile,
  * no injected failure leaves a role blocked at a rendezvous,
  * the model catches the hang of a relay that leaves early.
"""
import random
import threading

import pytest

WAIT_LIMIT_S = 0.05
HANG_S = 3.0
UNITS = [4, 1, 3, 2, 1, 5]  # steps (key tiles) of each query tile
K_SLOTS, V_SLOTS = 3, 2
UNIT_SLOTS = 4


class Hang(Exception):
    pass


class Rendezvous:
    """Named barrier over two warps returning the OR of their predicates."""

    def __init__(self):
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
                raise Hang(f"rendezvous generation {g}")
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
    def __init__(self, fail_p, seed, relay_leaves_early=False):
        self.rng = random.Random(seed)
        self.fail_p = fail_p
        self.early = relay_leaves_early
        self.lock = threading.Lock()
        self.abort = False
        self.q_full, self.q_empty = MBar(), MBar()
        self.k_full = [MBar() for _ in range(K_SLOTS)]
        self.k_empty = [MBar() for _ in range(K_SLOTS)]
        self.v_full = [MBar() for _ in range(V_SLOTS)]
        self.v_empty = [MBar() for _ in range(V_SLOTS)]
        self.s_full = [MBar(), MBar()]
        self.s_read, self.dp_full = MBar(2), MBar()
        self.ds_ready, self.dq_full, self.dq_free = MBar(2), MBar(), MBar(2)
        self.unit_full = [MBar() for _ in range(UNIT_SLOTS)]
        self.unit_empty = [MBar(4) for _ in range(UNIT_SLOTS)]  # issuer, relay, 2 warpgroups
        self.ring = [None] * UNIT_SLOTS
        self.next_unit = 0
        self.rv = Rendezvous()
        self.stored = 0

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


def publish(c, un):
    """Producer side of the unit ring: the next tile, or -1 after the last."""
    us = un % UNIT_SLOTS
    if not c.wait(c.unit_empty[us], ((un // UNIT_SLOTS) & 1) ^ 1):
        return None
    u = c.next_unit if c.next_unit < len(UNITS) else -1
    c.next_unit += 1
    c.ring[us] = u
    c.unit_full[us].arrive()
    return u


def read(c, un):
    us = un % UNIT_SLOTS
    u = c.ring[us]
    c.unit_empty[us].arrive()
    return u


def producer(c):
    k_it = v_it = 0
    un = q_it = 0
    while True:
        u = publish(c, un)
        un += 1
        if u is None or u < 0:
            return
        n = UNITS[u]
        if not c.wait(c.q_empty, (q_it & 1) ^ 1):
            return
        c.q_full.arrive()
        q_it += 1
        for _ in range(n):
            if not c.wait(c.k_empty[k_it % K_SLOTS], ((k_it // K_SLOTS) & 1) ^ 1):
                return
            c.k_full[k_it % K_SLOTS].arrive()
            k_it += 1
            if not c.wait(c.v_empty[v_it % V_SLOTS], ((v_it // V_SLOTS) & 1) ^ 1):
                return
            c.v_full[v_it % V_SLOTS].arrive()
            v_it += 1


def issuer(c):
    k_it = v_it = step = 0
    aborted = False
    un = 0
    while True:
        aborted = c.rv.go(aborted)                          # U
        if aborted:
            return
        u = read(c, un)
        un += 1
        if u < 0:
            return
        n = UNITS[u]
        prev_ks = 0
        for j in range(n):
            ks, vs, sb = k_it % K_SLOTS, v_it % V_SLOTS, step & 1
            aborted = c.rv.go(aborted)                      # A
            if not aborted:
                if j == 0:
                    c.q_empty.arrive()                     # copies of Q, dO done
                c.s_full[sb].arrive()
            if j > 0:
                aborted = c.rv.go(aborted)                  # B
                if not aborted:
                    c.k_empty[prev_ks].arrive()             # dQ += dS K_{j-1}
            aborted = c.rv.go(aborted)                      # C
            if not aborted:
                c.dp_full.arrive()
                c.v_empty[vs].arrive()
            prev_ks = ks
            k_it += 1
            v_it += 1
            step += 1
        aborted = c.rv.go(aborted)                          # D
        if not aborted:
            c.k_empty[prev_ks].arrive()
            c.dq_full.arrive()


def relay(c):
    k_it = v_it = step = 0
    aborted = False
    tile = 0  # tiles begun

    def wait(bar, parity):
        nonlocal aborted
        if not aborted:
            aborted = not c.wait(bar, parity)

    un = 0
    while True:
        wait(c.unit_full[un % UNIT_SLOTS], (un // UNIT_SLOTS) & 1)
        if aborted and c.early:
            return
        aborted = c.rv.go(aborted)                          # U
        if aborted:
            return
        u = read(c, un)
        un += 1
        if u < 0:
            return
        n = UNITS[u]
        for j in range(n):
            if j == 0:
                wait(c.q_full, tile & 1)
            wait(c.k_full[k_it % K_SLOTS], (k_it // K_SLOTS) & 1)
            if aborted and c.early:
                return
            aborted = c.rv.go(aborted)
            if j > 0:
                wait(c.ds_ready, (step - 1) & 1)
                if j == 1 and tile > 0:
                    wait(c.dq_free, (tile - 1) & 1)
                aborted = c.rv.go(aborted)
            wait(c.v_full[v_it % V_SLOTS], (v_it // V_SLOTS) & 1)
            wait(c.s_read, step & 1)
            aborted = c.rv.go(aborted)
            k_it += 1
            v_it += 1
            step += 1
        wait(c.ds_ready, (step - 1) & 1)
        if n == 1 and tile > 0:
            wait(c.dq_free, (tile - 1) & 1)
        aborted = c.rv.go(aborted)
        tile += 1


def warpgroup(c):
    step = 0
    tile = 0
    un = 0
    while True:
        us = un % UNIT_SLOTS
        if not c.wait(c.unit_full[us], (un // UNIT_SLOTS) & 1):
            return
        u = read(c, un)
        un += 1
        if u < 0:
            return
        for _ in range(UNITS[u]):
            if not c.wait(c.s_full[step & 1], (step >> 1) & 1):
                return
            c.s_read.arrive()
            if not c.wait(c.dp_full, step & 1):
                return
            c.ds_ready.arrive()
            step += 1
        if not c.wait(c.dq_full, tile & 1):
            return
        with c.lock:
            c.stored += 1
        c.dq_free.arrive()
        tile += 1


def run(fail_p, seed, relay_leaves_early=False):
    c = CTA(fail_p, seed, relay_leaves_early)
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
        th.join(4 * HANG_S)
    return c, hangs, sum(th.is_alive() for th in threads)


def test_clean_schedule_stores_every_tile():
    c, hangs, alive = run(0.0, 0)
    assert not hangs and alive == 0
    assert c.stored == 2 * len(UNITS)  # both warpgroups store their half of each tile


@pytest.mark.parametrize("seed", range(24))
def test_injected_wait_failures_never_hang(seed):
    fail_p = [0.005, 0.02, 0.1, 0.3][seed % 4]
    _, hangs, alive = run(fail_p, seed)
    assert not hangs and alive == 0, hangs


def test_model_catches_relay_that_leaves_early():
    found = False
    for seed in range(8):
        _, hangs, alive = run(0.3, 200 + seed, relay_leaves_early=True)
        if hangs or alive:
            found = True
            break
    assert found
