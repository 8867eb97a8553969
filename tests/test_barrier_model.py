"""CPU model of the persistent kernel's grid barrier (CPU only).

The protocol of `grid_sync`, transcribed to host threads: each CTA (thread) adds 1 to a
shared counter, then waits until the counter reaches epoch x grid; every wait polls a
deadline and the abort flag, and the first CTA to give up sets the abort flag and raises
MOE_ERR_TIMEOUT in the status word (compare-and-swap: the first error wins).  The device
implementation itself is covered by the GPU test that withholds one CTA's arrival; this
model checks the protocol's properties on many schedules without a GPU.
"""
import random
import threading
import time

MOE_ERR_TIMEOUT = -4


class Grid:
    def __init__(self, n):
        self.n = n
        self.bar = 0
        self.abort = 0
        self.status = [0, 0]
        self.lock = threading.Lock()
        self.arrivals = []   # (epoch, cta) in arrival order

    def atomic_add_bar(self, epoch, cta):
        with self.lock:
            self.bar += 1
            self.arrivals.append((epoch, cta))

    def atomic_exch_abort(self):
        with self.lock:
            old, self.abort = self.abort, 1
            return old

    def raise_status(self, code, detail):
        with self.lock:
            if self.status[0] == 0:
                self.status = [code, detail]


def grid_sync(g, cta, epoch, deadline, withhold=False):
    """One CTA's barrier: returns (ok, new_epoch)."""
    epoch += 1
    if not withhold:
        g.atomic_add_bar(epoch, cta)
    target = epoch * g.n
    spins = 0
    while g.bar < target:
        spins += 1
        if spins % 64 == 0 and (time.monotonic() > deadline or g.abort):
            if g.atomic_exch_abort() == 0:
                g.raise_status(MOE_ERR_TIMEOUT, -1)
            return False, epoch
        if spins % 256 == 0:
            time.sleep(0)
    return True, epoch


def _run(n, epochs, timeout_s, withhold_at=None, jitter=0.0, seed=0):
    g = Grid(n)
    results = [None] * n
    left_at = [[] for _ in range(n)]   # per CTA: counter value seen when leaving each barrier

    def cta(i):
        rng = random.Random(seed * 1000 + i)
        deadline = time.monotonic() + timeout_s
        epoch, ok_all, done = 0, True, 0
        for e in range(epochs):
            if jitter:
                time.sleep(rng.random() * jitter)
            ok, epoch = grid_sync(g, i, epoch, deadline, withhold=(withhold_at == (i, e)))
            if not ok:
                ok_all = False
                break
            left_at[i].append(g.bar)
            done += 1
        results[i] = (ok_all, done)

    ts = [threading.Thread(target=cta, args=(i,)) for i in range(n)]
    for t in ts:
        t.start()
    for t in ts:
        t.join(timeout=timeout_s + 30)
    assert not any(t.is_alive() for t in ts), "a barrier wait did not end"
    return g, results, left_at


def test_all_ctas_pass_every_epoch():
    n, epochs = 8, 40
    g, results, left_at = _run(n, epochs, timeout_s=20.0, jitter=0.0005, seed=1)
    assert all(r == (True, epochs) for r in results)
    assert g.bar == n * epochs and g.abort == 0 and g.status == [0, 0]
    # nobody leaves barrier e before every CTA has arrived at e
    for i in range(n):
        for e, seen in enumerate(left_at[i]):
            assert seen >= (e + 1) * n


def test_no_cta_runs_ahead_of_a_slow_one():
    n, epochs = 6, 25
    g, results, _ = _run(n, epochs, timeout_s=20.0, jitter=0.002, seed=2)
    assert all(ok for ok, _ in results)
    # arrivals for epoch e + 1 only start after every CTA arrived for epoch e
    last_of = {}
    first_of = {}
    for pos, (e, _) in enumerate(g.arrivals):
        last_of[e] = pos
        first_of.setdefault(e, pos)
    for e in range(1, epochs):
        assert first_of[e + 1] > last_of[e]


def test_a_withheld_arrival_times_out_every_cta_and_raises_once():
    n, epochs = 8, 10
    t0 = time.monotonic()
    g, results, _ = _run(n, epochs, timeout_s=0.5, withhold_at=(3, 4), seed=3)
    assert time.monotonic() - t0 < 10.0
    assert g.abort == 1
    assert g.status == [MOE_ERR_TIMEOUT, -1]
    for ok, done in results:   # every CTA passed epochs 0..3 and failed at epoch 4
        assert not ok and done == 4


def test_abort_flag_releases_waiters_before_their_deadline():
    n = 4
    g = Grid(n)
    out = {}

    def waiter(i):
        t = time.monotonic()
        ok, _ = grid_sync(g, i, 0, deadline=time.monotonic() + 60.0)
        out[i] = (ok, time.monotonic() - t)

    ts = [threading.Thread(target=waiter, args=(i,)) for i in range(n - 1)]   # one CTA never comes
    for t in ts:
        t.start()
    time.sleep(0.05)
    g.atomic_exch_abort()   # another wait elsewhere gave up
    for t in ts:
        t.join(timeout=30)
    assert all(not ok and dt < 30.0 for ok, dt in out.values())
    assert g.status == [0, 0]   # the CTA that set the flag raises the status, not the waiters
