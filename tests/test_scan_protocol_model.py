"""A CPU model of the synchronisation protocol of the lookahead scan kernel
(csrc/gdn_scan_la.cu), checked for deadlocks and stale reads (no GPU).

The model follows the kernel's barriers by name: B_SREADY (the 8 chain warps
publish the fp16 state image), B_YREADY (the key warps publish Y), B_MMA1 x3,
B_MMA2, B_MMA3 x2 (tensor-pipe commits).  mbarriers keep phase/parity
semantics, so a waiter that falls two phases behind blocks as it would on the
GPU; the tensor pipe runs the issued products in order; every buffer (the
MMA1 / MMA2 / MMA3 accumulators, the state image, the two Y buffers) carries
a version stamp, and every read asserts the version it must see.  The prep
images arrive in a three-slot ring (the image of chunk c + 1 is copied in once
MMA1(c) is done).  Random delays shake the interleavings.

Negative controls: the model must catch a product issued without its wait,
the MMA1 accumulator ring one buffer short, the MMA3 accumulator ring one
buffer short, and the prep-image ring one slot short.  In each, the warp or
product that would lose the race is held until the pipe has run the product
that races it (an event, not a sleep), so the bad interleaving is forced
whatever the load on the machine; in the protocol as built that product cannot
run first, and the hold ends on a short timeout."""
from __future__ import annotations

import queue
import random
import threading
import time

import pytest

TIMEOUT = 3.0


class _MBar:
    def __init__(self, count, name):
        self.count, self.pending, self.phase, self.name = count, count, 0, name
        self.cv = threading.Condition()

    def arrive(self):
        with self.cv:
            self.pending -= 1
            if self.pending == 0:
                self.phase += 1
                self.pending = self.count
                self.cv.notify_all()

    def wait(self, parity, who):
        # mbarrier.try_wait.parity: true once the phase of this parity has
        # completed, i.e. while the current phase has the other parity
        with self.cv:
            if not self.cv.wait_for(lambda: (self.phase & 1) != parity, timeout=TIMEOUT):
                raise RuntimeError(f"{who}: stuck on {self.name} (parity {parity})")


def _simulate(nch, *, n_d1=3, n_d3=2, n_p=3, wait_state_before_mma3=True, seed=0,
              query_delay=0.0, state_delay=0.0, hold=None, hold_timeout=0.05):
    """``hold``: (who, chunk) -- that party waits, before its racing access at
    that chunk, for the pipe to have run the product that races it:
    "state" (S_c's image write vs MMA3(c + 1)), "query_d1" (the read of O_{c-2}
    from D1 vs MMA1(c + 1)), "query_d3" (the same read from D3 vs MMA3(c)),
    "mma2" (MMA2(c)'s read of the prep image vs the copy of image c + 1)."""
    rnd = random.Random(seed)
    lock = threading.Lock()
    buf = {}
    errors = []
    done = {}  # events: products run by the pipe, images copied in

    def event(key):
        with lock:
            if key not in done:
                done[key] = threading.Event()
            return done[key]

    def release_all():
        with lock:
            evs = list(done.values())
        for ev in evs:
            ev.set()

    def held(who, c, key):
        # in the protocol as built the racing product cannot run first, and
        # the wait ends on its timeout
        if hold == (who, c):
            event(key).wait(timeout=hold_timeout)

    def jitter():
        if rnd.random() < 0.3:
            time.sleep(rnd.random() * 3e-4)

    def write(key, tag):
        with lock:
            buf[key] = tag

    def read(key, want, who):
        with lock:
            got = buf.get(key)
        if got != want:
            raise AssertionError(f"{who}: {key} holds {got}, expected {want}")

    bars = {"SREADY": _MBar(8, "B_SREADY"), "YREADY": _MBar(4, "B_YREADY"),
            "MMA2": _MBar(1, "B_MMA2")}
    bars.update({f"MMA1_{i}": _MBar(1, f"B_MMA1+{i}") for i in range(n_d1)})
    bars.update({f"MMA3_{i}": _MBar(1, f"B_MMA3+{i}") for i in range(n_d3)})
    d1 = lambda c: c % n_d1                       # noqa: E731
    d3 = lambda e: (e - 1) % n_d3                 # noqa: E731
    d1_parity = lambda c: ((c - 1) // n_d1) & 1   # noqa: E731  (MMA1(0) does not exist)
    d3_parity = lambda e: (e // n_d3) & 1         # noqa: E731  (MMA3(0) is the first)
    pipe = queue.Queue()

    def pipe_worker():
        ok = True
        while True:
            op = pipe.get()
            if op is None:
                return
            if ok:
                try:
                    jitter()
                    op()
                except Exception as e:  # noqa: BLE001
                    errors.append(e)
                    ok = False
                    release_all()

    def commit(name):
        pipe.put(lambda: bars[name].arrive())

    def copy_image(j):  # the prep image of chunk j into slot j % n_p
        write(("P", j % n_p), ("P", j))
        event(("P", j)).set()

    def mma1(c):  # [E_c; AqkT_{c-1}] Y_{c-1}
        def op():
            read(("Y", (c - 1) & 1), ("Y", c - 1), f"MMA1({c})")
            read(("P", (c - 1) % n_p), ("P", c - 1), f"MMA1({c})")
            write(("D1", d1(c)), ("MMA1", c))
            event(("MMA1", c)).set()
        pipe.put(op)
        commit(f"MMA1_{d1(c)}")

    def mma2(c):  # P1_{c-1} Y_{c-1}: the state update
        def op():
            held("mma2", c, ("P", c + 1))
            read(("Y", (c - 1) & 1), ("Y", c - 1), f"MMA2({c})")
            read(("P", (c - 1) % n_p), ("P", c - 1), f"MMA2({c})")
            write("D2", ("MMA2", c))
        pipe.put(op)
        commit("MMA2")

    def mma3(e):  # [K_e; Q_{e-1}] S_{e-1} (e = 0: [K_0; Q_0] S_0)
        def op():
            read("S", ("S", max(e - 1, 0)), f"MMA3({e})")
            write(("D3", d3(e)), ("MMA3", e))
            event(("MMA3", e)).set()
        pipe.put(op)
        commit(f"MMA3_{d3(e)}")

    def issuer():
        try:
            copy_image(0)
            if nch > 1:
                copy_image(1)
            bars["SREADY"].wait(0, "issuer: S_0")
            mma3(0)
            for c in range(1, nch + 1):
                jitter()
                bars["YREADY"].wait((c - 1) & 1, f"issuer: Y_{c - 1}")
                mma1(c)
                if wait_state_before_mma3:
                    bars["SREADY"].wait((c - 1) & 1, f"issuer: S_{c - 1}")
                mma3(c)
                mma2(c)
                # the image of chunk c + 1 into the slot of chunk c - 2 once
                # MMA1(c) is done (the pipe runs in order: MMA2(c - 1), that
                # slot's last reader, is done too)
                if c + 1 < nch:
                    bars[f"MMA1_{d1(c)}"].wait(d1_parity(c), f"issuer: MMA1({c})")
                    copy_image(c + 1)
        except Exception as e:  # noqa: BLE001
            errors.append(e)
        finally:
            pipe.put(None)

    def chain(w):
        q = w & 3
        key, query = q < 2, q >= 2  # C = 64: lanes 0-63 keys, 64-127 queries
        try:
            if w == 0:
                write("S", ("S", 0))
            bars["SREADY"].arrive()
            for c in range(nch + 1):
                jitter()
                if query and c >= 2:  # deferred output of chunk c - 2
                    time.sleep(query_delay)
                    held("query_d3", c, ("MMA3", c))
                    read(("D3", d3(c - 1)), ("MMA3", c - 1), f"warp {w}: O_{c - 2}")
                    held("query_d1", c, ("MMA1", c + 1))
                    read(("D1", d1(c - 1)), ("MMA1", c - 1), f"warp {w}: O_{c - 2}")
                if c >= 1:
                    bars[f"MMA1_{d1(c)}"].wait(d1_parity(c), f"warp {w}: MMA1({c})")
                bars[f"MMA3_{d3(c)}"].wait(d3_parity(c), f"warp {w}: MMA3({c})")
                if key and c < nch:
                    read(("D3", d3(c)), ("MMA3", c), f"warp {w}: X_{c}")
                    if c >= 1:
                        read(("D1", d1(c)), ("MMA1", c), f"warp {w}: X_{c}")
                    jitter()
                    if w == 0:
                        write(("Y", c & 1), ("Y", c))
                    bars["YREADY"].arrive()
                if c >= 1:  # the state after Y_c: S_c = d S_{c-1} + MMA2(c)
                    bars["MMA2"].wait((c - 1) & 1, f"warp {w}: MMA2({c})")
                    read("D2", ("MMA2", c), f"warp {w}: S_{c}")
                    if c < nch:
                        if w == 0:
                            time.sleep(state_delay)
                            held("state", c, ("MMA3", c + 1))
                            write("S", ("S", c))
                        bars["SREADY"].arrive()
            if query:
                read(("D3", d3(nch)), ("MMA3", nch), f"warp {w}: O_{nch - 1}")
                read(("D1", d1(nch)), ("MMA1", nch), f"warp {w}: O_{nch - 1}")
        except Exception as e:  # noqa: BLE001
            errors.append(e)

    threads = [threading.Thread(target=pipe_worker, daemon=True),
               threading.Thread(target=issuer, daemon=True)]
    threads += [threading.Thread(target=chain, args=(w,), daemon=True) for w in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=4 * TIMEOUT)
    if not errors and any(t.is_alive() for t in threads):
        errors.append(RuntimeError("threads still running"))
    return errors


@pytest.mark.parametrize("nch", [1, 2, 3, 4, 7, 12])
def test_protocol_as_built_has_no_deadlock_or_stale_read(nch):
    for seed in range(12):
        errors = _simulate(nch, seed=seed)
        assert not errors, f"seed {seed}: {errors[0]}"


@pytest.mark.parametrize("slow", ["query", "state"])
def test_protocol_as_built_tolerates_late_warps(slow):
    """Late query warps (the deferred output) or a late state image must only
    slow the chain down, never let a product overwrite what they still read."""
    kw = {"query_delay": 2e-3} if slow == "query" else {"state_delay": 2e-3}
    errors = _simulate(7, **kw)
    assert not errors, errors[0]


@pytest.mark.parametrize("hold", ["state", "query_d1", "query_d3", "mma2"])
def test_protocol_as_built_survives_every_forced_hold(hold):
    """The holds of the negative controls, on the protocol as built: each
    racing product cannot run first, so every hold only ends on its timeout."""
    for c in (2, 3):
        errors = _simulate(6, hold=(hold, c))
        assert not errors, f"hold {hold} at chunk {c}: {errors[0]}"


def _caught(hold, **mutation):
    # the held party waits for the racing product (an event), so the race
    # happens whatever the machine's load; chunks 2 and 3 are both tried
    return all(_simulate(6, hold=(hold, c), hold_timeout=2.0, **mutation) for c in (2, 3))


def test_model_catches_a_product_issued_without_its_wait():
    # MMA3(c + 1) sent without waiting for S_c's image
    assert _caught("state", wait_state_before_mma3=False)


def test_model_catches_an_mma1_accumulator_ring_one_buffer_short():
    # the query lanes read MMA1's accumulator one chunk late, which is why the
    # kernel keeps three of them: with two, MMA1(c + 1) overwrites it first
    assert _caught("query_d1", n_d1=2)


def test_model_catches_an_mma3_accumulator_ring_one_buffer_short():
    # with one MMA3 accumulator, MMA3(c) overwrites what O_{c-2} still reads
    assert _caught("query_d3", n_d3=1)


def test_model_catches_a_prep_image_ring_one_slot_short():
    # with two slots, the image of chunk c + 1 lands in the slot MMA2(c)
    # still reads (waiting for MMA1(c) does not cover MMA2(c))
    assert _caught("mma2", n_p=2)
