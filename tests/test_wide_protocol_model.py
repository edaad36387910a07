"""Host models of the wide-head-dim kernels' coordination protocols (no GPU).

The d in {192, 256} kernels keep the abort rule of the narrower ones: after a
bounded mbarrier wait runs out, the roles that meet at named barriers (which
have no time limit) walk their schedules to the end with waits and work
skipped, so every barrier generation still pairs up.  These models run the
roles as threads with the kernels' loop structure -- the forward's one query
tile per unit with two S buffers, its K/V chunk ring in consumption order
(K0 K1 V0 K2 V1 ...) and its P V completion barrier waited only on a rescale;
the backward's dK/dV kernel (64-row Q/dO items through a ring, the unit's K
halves through the same ring, units handed out at run time through a
4-entry ring after which the relay and issuer leave together at the next
unit's rendezvous once aborted) and dQ kernel (Q halves and K_j/V_j items) --
with named barriers as OR-reducing rendezvous and mbarriers as phase counters
whose waits fail at randomly injected points, and check that no injected
failure leaves a role blocked, that a clean run completes every epilogue,
and that the models catch a role that leaves early.
"""
import random
import threading

import pytest

from test_fwd_protocol_model import Hang, MBar, Rendezvous

WAIT_LIMIT_S = 0.05
HANG_S = 3.0


class Ctx:
    """Shared state of one modelled CTA: injected failures and the abort flag."""

    def __init__(self, fail_p, seed, rescale_p=0.0):
        self.rng = random.Random(seed)
        self.fail_p, self.rescale_p = fail_p, rescale_p
        self.lock = threading.Lock()
        self.abort = False
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

    def coin(self, p):
        with self.lock:
            return self.rng.random() < p


def run_roles(roles, c):
    hangs = []

    def wrap(f, *a):
        try:
            f(c, *a)
        except Hang as e:
            hangs.append(str(e))

    threads = [threading.Thread(target=wrap, args=(f,) + a, daemon=True) for f, a in roles]
    for th in threads:
        th.start()
    for th in threads:
        th.join(4 * HANG_S)
    return hangs, sum(th.is_alive() for th in threads)


# ------------------------------------------------------------- wide forward ---

FWD_UNITS = [3, 1, 5, 2, 4, 1, 6]  # key blocks of each unit's query tile
CH, RING = 4, 10                   # chunks per K or V tile, ring depth (d = 256)


def tile_order(nb):
    """K0 K1 V0 K2 V1 K3 ... V(nb-1), as the kernel's for_each_tile."""
    seq = [("K", 0)] + ([("K", 1)] if nb > 1 else [])
    for j in range(nb):
        seq.append(("V", j))
        if j + 2 < nb:
            seq.append(("K", j + 2))
    return seq


class Fwd(Ctx):
    def __init__(self, fail_p, seed, rescale_p=0.0, early=False):
        super().__init__(fail_p, seed, rescale_p)
        self.early = early
        self.qfull, self.qempty = MBar(), MBar()
        self.sfull = [MBar(), MBar()]
        self.pvdone, self.ofull = MBar(), MBar()
        self.kvfull = [MBar() for _ in range(RING)]
        self.kvempty = [MBar() for _ in range(RING)]
        self.kv, self.p = Rendezvous("kBarKv"), Rendezvous("kBarP")


def fwd_producer(c):
    it = q_it = 0
    for nb in FWD_UNITS:
        if not c.wait(c.qempty, (q_it & 1) ^ 1):
            return
        c.qfull.arrive()
        q_it += 1
        for _ in tile_order(nb):
            for _ in range(CH):
                slot = it % RING
                if not c.wait(c.kvempty[slot], ((it // RING) & 1) ^ 1):
                    return
                c.kvfull[slot].arrive()
                it += 1


def fwd_relay(c):
    it = q_it = 0
    aborted = False

    def tile_ready():
        nonlocal it, aborted
        for _ in range(CH):
            slot, par = it % RING, (it // RING) & 1
            it += 1
            if not aborted:
                aborted = not c.wait(c.kvfull[slot], par)

    for nb in FWD_UNITS:
        par = q_it & 1
        q_it += 1
        if not aborted:
            aborted = not c.wait(c.qfull, par)
        tile_ready()
        aborted = c.kv.go(aborted)
        if nb > 1:
            tile_ready()
            aborted = c.kv.go(aborted)
        for j in range(nb):
            tile_ready()
            if j + 2 < nb:
                tile_ready()
            aborted = c.kv.go(aborted)


def fwd_issuer(c):
    it = s_it = 0
    aborted = False

    def release(pos):
        for x in range(CH):
            c.kvempty[(pos + x) % RING].arrive()

    for nb in FWD_UNITS:
        s0 = s_it
        aborted = c.kv.go(aborted)
        k0 = it
        it += CH
        if not aborted:
            c.sfull[s0 & 1].arrive()
            release(k0)
            if nb == 1:
                c.qempty.arrive()
        if nb > 1:
            aborted = c.kv.go(aborted)
            k1 = it
            it += CH
            if not aborted:
                c.sfull[(s0 + 1) & 1].arrive()
                release(k1)
                if nb == 2:
                    c.qempty.arrive()
        for j in range(nb):
            aborted = c.kv.go(aborted)
            vpos = it
            it += CH
            nxt = j + 2 < nb
            k2 = 0
            if nxt:
                k2 = it
                it += CH
            aborted = c.p.go(aborted)
            if not aborted:
                c.pvdone.arrive()
                release(vpos)
                if j == nb - 1:
                    c.ofull.arrive()
                if nxt:
                    c.sfull[(s0 + j) & 1].arrive()
                    release(k2)
                    if j + 2 == nb - 1:
                        c.qempty.arrive()
        s_it += nb


def fwd_softmax(c):
    s_it = o_it = pv_it = 0
    aborted = False
    for nb in FWD_UNITS:
        for j in range(nb):
            sidx = s_it + j
            if not aborted:
                aborted = not c.wait(c.sfull[sidx & 1], (sidx >> 1) & 1)
            if aborted and c.early:
                return
            if not aborted and j > 0 and c.coin(c.rescale_p):
                # the rescale waits for P V(j-1)
                aborted = not c.wait(c.pvdone, (pv_it + j - 1) & 1)
            aborted = c.p.go(aborted)
        s_it += nb
        pv_it += nb
        par = o_it & 1
        o_it += 1
        if not aborted:
            aborted = not c.wait(c.ofull, par)
        if not aborted:
            with c.lock:
                c.epilogues += 1


def run_fwd(fail_p, seed, rescale_p=0.0, early=False):
    c = Fwd(fail_p, seed, rescale_p, early)
    hangs, alive = run_roles([(fwd_producer, ()), (fwd_relay, ()), (fwd_issuer, ()),
                              (fwd_softmax, ())], c)
    return c, hangs, alive


def test_wide_forward_clean_schedule():
    c, hangs, alive = run_fwd(0.0, 0, rescale_p=0.5)
    assert not hangs and alive == 0
    assert c.epilogues == len(FWD_UNITS)


@pytest.mark.parametrize("seed", range(16))
def test_wide_forward_injected_failures_never_hang(seed):
    fail_p = [0.005, 0.02, 0.1, 0.3][seed % 4]
    _, hangs, alive = run_fwd(fail_p, seed, rescale_p=[0.0, 0.5, 1.0][seed % 3])
    assert not hangs and alive == 0, hangs


def test_wide_forward_model_catches_softmax_that_leaves_early():
    assert any(run_fwd(0.3, 50 + s, early=True)[1:] != ([], 0) for s in range(6))


# ----------------------------------------------------------- wide backward ---
# Both wide backward kernels pair only the issuer and the relay at a named
# barrier; the compute warpgroups and the producer leave at their first failed
# wait.  The model follows the dK/dV kernel's schedule, per step the
# rendezvous [Q_i (+ K, V at the unit's start)] [dS of the previous step]
# [dO_i] [P (+ dK, dV stored at the unit's start)], then the unit's last dK;
# the dQ kernel's ([K_j (+ Q, dO)] [dS_{j-1} (+ dQ free)] [V_j, S_j read],
# then the last dQ) has the same shape with one rendezvous fewer per step.

BWD_UNITS = [4, 1, 3, 2, 5]  # steps of each unit
R = 5                        # ring slots
UNIT_SLOTS = 4               # unit ring entries


class Bwd(Ctx):
    def __init__(self, fail_p, seed, k_halves, early=False):
        super().__init__(fail_p, seed)
        self.k_halves = k_halves  # ring items a unit takes before its steps
        self.early = early
        self.tilefull, self.tileempty = MBar(), MBar()  # resident tiles (V, or Q/dO staging)
        self.full = [MBar() for _ in range(R)]
        self.empty = [MBar() for _ in range(R)]
        self.sfull, self.dpfull = MBar(), MBar()
        self.pready, self.dsready = MBar(), MBar()
        self.outfull, self.outfree = MBar(), MBar()
        self.relay_bar = Rendezvous("kBarRelay")
        self.unit_full = [MBar() for _ in range(UNIT_SLOTS)]
        self.unit_empty = [MBar(3) for _ in range(UNIT_SLOTS)]  # relay, issuer, compute
        self.ring_units = [None] * UNIT_SLOTS
        self.next_unit = 0


def bwd_publish(c, un):
    us = un % UNIT_SLOTS
    if not c.wait(c.unit_empty[us], ((un // UNIT_SLOTS) & 1) ^ 1):
        return None
    u = c.next_unit if c.next_unit < len(BWD_UNITS) else -1
    c.next_unit += 1
    c.ring_units[us] = u
    c.unit_full[us].arrive()
    return u


def bwd_read_unit(c, un):
    us = un % UNIT_SLOTS
    u = c.ring_units[us]
    c.unit_empty[us].arrive()
    return u


def bwd_producer(c):
    it = unit_it = un = 0
    while True:
        u = bwd_publish(c, un)
        un += 1
        if u is None or u < 0:
            return
        steps = BWD_UNITS[u]
        if not c.wait(c.tileempty, (unit_it & 1) ^ 1):
            return
        c.tilefull.arrive()
        unit_it += 1
        for _ in range(c.k_halves + 2 * steps):
            if not c.wait(c.empty[it % R], ((it // R) & 1) ^ 1):
                return
            c.full[it % R].arrive()
            it += 1


def bwd_relay(c):
    it = st_it = unit_it = 0
    aborted = False

    def wait_all(bar, par):
        nonlocal aborted
        if not aborted:
            aborted = not c.wait(bar, par)

    un = 0
    while True:
        wait_all(c.unit_full[un % UNIT_SLOTS], (un // UNIT_SLOTS) & 1)
        aborted = c.relay_bar.go(aborted)
        if aborted:
            return
        u = bwd_read_unit(c, un)
        un += 1
        if u < 0:
            return
        steps = BWD_UNITS[u]
        wait_all(c.tilefull, unit_it & 1)
        for _ in range(c.k_halves):
            wait_all(c.full[it % R], (it // R) & 1)
            it += 1
        for s in range(steps):
            a, b = it, it + 1
            it += 2
            par = st_it & 1
            wait_all(c.full[a % R], (a // R) & 1)
            aborted = c.relay_bar.go(aborted)
            if s > 0:
                wait_all(c.dsready, par ^ 1)
                aborted = c.relay_bar.go(aborted)
            wait_all(c.full[b % R], (b // R) & 1)
            aborted = c.relay_bar.go(aborted)
            if s == 0 and unit_it > 0:
                wait_all(c.outfree, (unit_it - 1) & 1)
            wait_all(c.pready, par)
            aborted = c.relay_bar.go(aborted)
            st_it += 1
        wait_all(c.dsready, (st_it - 1) & 1)
        aborted = c.relay_bar.go(aborted)
        unit_it += 1


def bwd_issuer(c):
    it = un = 0
    aborted = False
    while True:
        aborted = c.relay_bar.go(aborted)
        if aborted:
            return
        u = bwd_read_unit(c, un)
        un += 1
        if u < 0:
            return
        steps = BWD_UNITS[u]
        kpos = it
        it += c.k_halves
        prev = None
        for s in range(steps):
            a, b = it, it + 1
            it += 2
            aborted = c.relay_bar.go(aborted)
            if not aborted:
                if s == 0:
                    for x in range(c.k_halves):  # copied to tensor memory, released
                        c.empty[(kpos + x) % R].arrive()
                c.sfull.arrive()
            if s > 0:
                aborted = c.relay_bar.go(aborted)
                if not aborted:
                    c.empty[prev[0] % R].arrive()
                    c.empty[prev[1] % R].arrive()
            aborted = c.relay_bar.go(aborted)
            if not aborted:
                c.dpfull.arrive()
                if s == steps - 1:
                    c.tileempty.arrive()
            aborted = c.relay_bar.go(aborted)
            prev = (a, b)
        aborted = c.relay_bar.go(aborted)
        if not aborted:
            c.empty[prev[0] % R].arrive()
            c.empty[prev[1] % R].arrive()
            c.outfull.arrive()


def bwd_compute(c):
    st_it = unit_it = un = 0
    while True:
        if not c.wait(c.unit_full[un % UNIT_SLOTS], (un // UNIT_SLOTS) & 1):
            return
        u = bwd_read_unit(c, un)
        un += 1
        if u < 0:
            return
        steps = BWD_UNITS[u]
        for _ in range(steps):
            par = st_it & 1
            if not c.wait(c.sfull, par):
                return
            if c.early and c.coin(0.3):
                return
            c.pready.arrive()
            if not c.wait(c.dpfull, par):
                return
            c.dsready.arrive()
            st_it += 1
        if not c.wait(c.outfull, unit_it & 1):
            return
        unit_it += 1
        c.outfree.arrive()
        with c.lock:
            c.epilogues += 1


def run_bwd(fail_p, seed, k_halves, early=False):
    c = Bwd(fail_p, seed, k_halves, early)
    hangs, alive = run_roles([(bwd_producer, ()), (bwd_relay, ()), (bwd_issuer, ()),
                              (bwd_compute, ())], c)
    return c, hangs, alive


@pytest.mark.parametrize("k_halves", [0, 2])  # d = 192 (K resident), d = 256 (K via the ring)
def test_wide_backward_clean_schedule(k_halves):
    c, hangs, alive = run_bwd(0.0, 0, k_halves)
    assert not hangs and alive == 0
    assert c.epilogues == len(BWD_UNITS)


@pytest.mark.parametrize("k_halves", [0, 2])
@pytest.mark.parametrize("seed", range(12))
def test_wide_backward_injected_failures_never_hang(k_halves, seed):
    fail_p = [0.005, 0.02, 0.1, 0.3][seed % 4]
    _, hangs, alive = run_bwd(fail_p, 100 + seed, k_halves)
    assert not hangs and alive == 0, hangs
