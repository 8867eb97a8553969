"""CPU model of the persistent kernel's grid barrier (CPU only).

The protocol of `grid_arrive` / `grid_wait`, transcribed to host threads: one 32-bit word
serves every barrier of every launch.  Each CTA adds 1 to it, except CTA 0, which adds
2^31 - (G - 1); the G additions of one barrier sum to 2^31, so the low 31 bits return to 0
and bit 31 flips, and only with the last addition.  A CTA remembers the value its own
addition returned and waits until bit 31 of the word differs from it.  Every wait polls a
deadline and the abort flag, and the first CTA to give up sets the abort flag and raises
MOE_ERR_TIMEOUT in the status word (compare-and-swap: the first error wins).  The device
implementation itself is covered by the GPU tests that withhold one CTA's arrival; this
model checks the protocol's properties on many schedules without a GPU.
"""
import itertools
import random
import threading
import time

MOE_ERR_TIMEOUT = -4
MASK = (1 << 32) - 1
BIT31 = 1 << 31


class Grid:
    def __init__(self, n, word=0):
        self.n = n
        self.bar = word   # the barrier word (at rest: low 31 bits 0; bit 31 either way)
        self.abort = 0
        self.status = [0, 0]
        self.lock = threading.Lock()
        self.arrivals = []   # (barrier, cta) in arrival order
        self.passes = 0      # barriers completed (bit-31 flips)

    def atomic_add_bar(self, add, barrier, cta):
        with self.lock:
            old = self.bar
            self.bar = (self.bar + add) & MASK
            if (old ^ self.bar) & BIT31:
                self.passes += 1
            self.arrivals.append((barrier, cta))
            return old

    def load_bar(self):
        with self.lock:
            return self.bar

    def atomic_exch_abort(self):
        with self.lock:
            old, self.abort = self.abort, 1
            return old

    def raise_status(self, code, detail):
        with self.lock:
            if self.status[0] == 0:
                self.status = [code, detail]


def grid_sync(g, cta, barrier, deadline, withhold=False):
    """One CTA's barrier number `barrier`: returns ok."""
    add = (BIT31 - (g.n - 1)) & MASK if cta == 0 else 1
    token = g.load_bar() if withhold else g.atomic_add_bar(add, barrier, cta)
    spins = 0
    while not ((g.load_bar() ^ token) & BIT31):
        spins += 1
        if spins % 64 == 0 and (time.monotonic() > deadline or g.abort):
            if g.atomic_exch_abort() == 0:
                g.raise_status(MOE_ERR_TIMEOUT, -1)
            return False
        if spins % 256 == 0:
            time.sleep(0)
    return True


def _run(n, epochs, timeout_s, withhold_at=None, jitter=0.0, seed=0, g=None):
    g = Grid(n) if g is None else g
    results = [None] * n
    left_at = [[] for _ in range(n)]   # per CTA: barriers completed when it left each barrier

    def cta(i):
        rng = random.Random(seed * 1000 + i)
        deadline = time.monotonic() + timeout_s
        ok_all, done = True, 0
        for e in range(epochs):
            if jitter:
                time.sleep(rng.random() * jitter)
            ok = grid_sync(g, i, e, deadline, withhold=(withhold_at == (i, e)))
            if not ok:
                ok_all = False
                break
            left_at[i].append(g.passes)
            done += 1
        results[i] = (ok_all, done)

    ts = [threading.Thread(target=cta, args=(i,)) for i in range(n)]
    for t in ts:
        t.start()
    for t in ts:
        t.join(timeout=timeout_s + 30)
    assert not any(t.is_alive() for t in ts), "a barrier wait did not end"
    return g, results, left_at


def test_bit31_flips_only_with_the_last_addition_in_every_order():
    """Exhaustive over arrival orders (G <= 6) and both resting values of bit 31."""
    for n in range(1, 7):
        for word in (0, BIT31):
            for order in itertools.permutations(range(n)):
                v = word
                for pos, cta in enumerate(order):
                    add = (BIT31 - (n - 1)) & MASK if cta == 0 else 1
                    old, v = v, (v + add) & MASK
                    assert (old & BIT31) == (word & BIT31)   # every token carries the barrier's bit
                    flipped = (v ^ word) & BIT31
                    assert bool(flipped) == (pos == n - 1), (n, order, pos)
                assert v == word ^ BIT31   # at rest again: low 31 bits 0, bit 31 flipped


def test_all_ctas_pass_every_epoch():
    n, epochs = 8, 40
    g, results, left_at = _run(n, epochs, timeout_s=20.0, jitter=0.0005, seed=1)
    assert all(r == (True, epochs) for r in results)
    assert g.passes == epochs and g.abort == 0 and g.status == [0, 0]
    assert g.bar & (BIT31 - 1) == 0   # the word is back at rest
    # nobody leaves barrier e before every CTA has arrived at e (barrier e completed)
    for i in range(n):
        for e, seen in enumerate(left_at[i]):
            assert seen >= e + 1


def test_consecutive_launches_reuse_the_word_without_clearing():
    n, epochs = 5, 7
    g = Grid(n)
    for launch in range(4):   # 7 barriers each: bit 31 ends flipped on odd counts
        g.arrivals = []
        _, results, _ = _run(n, epochs, timeout_s=20.0, jitter=0.0003, seed=10 + launch, g=g)
        assert all(r == (True, epochs) for r in results)
        assert g.bar & (BIT31 - 1) == 0
    assert g.passes == 4 * epochs


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
    for e in range(epochs - 1):
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
        ok = grid_sync(g, i, 0, deadline=time.monotonic() + 60.0)
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
