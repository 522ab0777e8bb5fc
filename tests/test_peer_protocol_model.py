"""A CPU model of the multi-GPU all-reduce's protocol (ar_allreduce_peer), checked on threads.

Each rank's kernel has B blocks; here every (rank, block) is a thread, and a
rank's threads meet at a barrier at the end of every call (the kernel
boundary: the next call on a rank's stream starts after the previous kernel).
Every rank holds flag words flags[ph][b][src] and two data areas; call e uses
area e & 1.  Block b of rank r, in call e:

  one-shot:  copy its range of the input into its area; barrier 0; sum the
             range over every rank's area (rank order) into out.
  two-shot:  copy part b of every rank slice into its area; barrier 0; sum
             part b of its own slice over every rank's area into out and back
             into its area; barrier 1; copy part b of every other slice from
             that slice's rank into out.
  barrier ph: store e into flags[ph][b][r] of every rank; wait (bounded)
             until its own flags[ph][b][t] >= e for every rank t.

The model checks, over random timings: every rank gets the exact sum in every
call; every element a block reads from an area holds the data of the call it
reads for, never an earlier or a later call's (the reason for the two areas:
each element carries the call that wrote it); and a rank that stops making
calls makes the others' waits run out instead of hang.  A variant with one
data area shows that the check has teeth.
"""
import random
import threading
import time

import pytest

WAIT_S = 1.0


class Hazard(AssertionError):
    pass


class World:
    def __init__(self, R, B, n, areas=2, seed=0, slow=None):
        self.R, self.B, self.n, self.areas = R, B, n, areas
        self.rng = random.Random(seed)
        self.flags = [[[[0] * R for _ in range(B)] for _ in range(2)] for _ in range(R)]
        self.data = [[[None] * n for _ in range(areas)] for _ in range(R)]
        self.lock = threading.Lock()
        self.timeouts = 0
        self.errors = []
        self.slow = slow or {}

    def pause(self, r):
        time.sleep(self.rng.random() * 0.0004 * self.slow.get(r, 1.0))

    # -- reading and writing an area: every element carries the call that wrote it
    def write(self, r, area, idx, e, value):
        self.data[r][area][idx] = (e, value)

    def read(self, q, area, idx, e, reader):
        w_e, value = self.data[q][area][idx]
        if w_e != e:
            raise Hazard(f"rank {reader} read element {idx} of rank {q}'s area {area} in call {e}, "
                         f"but it holds call {w_e}'s data")
        return value

    # -- the per-block barrier
    def barrier(self, r, b, ph, e):
        for t in range(self.R):
            self.flags[t][ph][b][r] = e
            self.pause(r)
        t0 = time.monotonic()
        for t in range(self.R):
            while self.flags[r][ph][b][t] < e:
                if time.monotonic() - t0 > WAIT_S:
                    with self.lock:
                        self.timeouts += 1
                    return False
                time.sleep(0.0001)
        return True


def block_range(n, B, b):
    per = -(-n // B)
    return range(min(n, b * per), min(n, (b + 1) * per))


def two_shot_part(n, R, B, s, b):
    slice_ = -(-n // R)
    s0, s1 = min(n, s * slice_), min(n, (s + 1) * slice_)
    per = -(-(s1 - s0) // B)
    return range(min(s1, s0 + b * per), min(s1, s0 + (b + 1) * per))


def run_block(w, r, b, calls, inputs, outs, twoshot, kernel_end, stop_after):
    R, B, n = w.R, w.B, w.n
    for e in range(1, calls + 1):
        if r in stop_after and e > stop_after[r]:
            return
        area = e % w.areas
        x, out = inputs[r][e], outs[r][e]
        mine = [block_range(n, B, b)] if not twoshot else [two_shot_part(n, R, B, s, b) for s in range(R)]
        for rng_ in mine:                                     # copy into this rank's area
            for i in rng_:
                w.write(r, area, i, e, x[i])
            w.pause(r)
        if w.barrier(r, b, 0, e):
            own = block_range(n, B, b) if not twoshot else two_shot_part(n, R, B, r, b)
            for i in own:                                     # rank-order sum
                terms = []
                for q in range(R):
                    terms.append(w.read(q, area, i, e, r))
                    w.pause(r)
                out[i] = sum(terms)
            if twoshot:
                for i in own:                                 # the reduced part, for the peers' gather
                    w.write(r, area, i, e, out[i])
                if w.barrier(r, b, 1, e):
                    for s in range(R):
                        if s == r:
                            continue
                        for i in two_shot_part(n, R, B, s, b):
                            out[i] = w.read(s, area, i, e, r)
                            w.pause(r)
        try:
            kernel_end[r].wait(timeout=10)                    # the next call starts after this kernel
        except threading.BrokenBarrierError:
            return


def simulate(R, B, n, calls, twoshot, seed, areas=2, stop_after=None, slow=None):
    rng = random.Random(seed)
    w = World(R, B, n, areas=areas, seed=seed, slow=slow)
    stop_after = stop_after or {}
    inputs = [[None] + [[rng.randint(-1000, 1000) for _ in range(n)] for _ in range(calls)] for _ in range(R)]
    outs = [[None] + [[None] * n for _ in range(calls)] for _ in range(R)]
    kernel_end = [threading.Barrier(B) for _ in range(R)]
    threads = []
    for r in range(R):
        for b in range(B):
            def body(r=r, b=b):
                try:
                    run_block(w, r, b, calls, inputs, outs, twoshot, kernel_end, stop_after)
                except Hazard as h:
                    w.errors.append(h)
                    for kb in kernel_end:
                        kb.abort()
            t = threading.Thread(target=body, daemon=True)
            threads.append(t)
            t.start()
    for t in threads:
        t.join(timeout=60)
        assert not t.is_alive(), "a block never finished: the protocol hangs"
    return w, inputs, outs


@pytest.mark.parametrize("twoshot", [False, True])
def test_every_rank_gets_the_exact_sum_in_every_call(twoshot):
    for seed in range(6):
        R, B, n, calls = random.Random(seed).choice([(2, 2, 13), (3, 2, 40), (4, 3, 31)]) + (5,)
        w, inputs, outs = simulate(R, B, n, calls, twoshot, seed)
        assert not w.errors, w.errors
        assert w.timeouts == 0
        for e in range(1, calls + 1):
            want = [sum(inputs[q][e][i] for q in range(R)) for i in range(n)]
            for r in range(R):
                assert outs[r][e] == want, (seed, r, e)


@pytest.mark.parametrize("twoshot", [False, True])
def test_a_rank_that_stops_makes_the_others_time_out(twoshot):
    """Rank 2 makes two calls of four: the other ranks' third call waits for it, gives up after the
    bounded wait, and every thread ends (no hang); the first two calls are exact."""
    R, B, n = 3, 2, 20
    w, inputs, outs = simulate(R, B, n, 4, twoshot, seed=5, stop_after={2: 2})
    assert not w.errors
    assert w.timeouts > 0
    for e in (1, 2):
        want = [sum(inputs[q][e][i] for q in range(R)) for i in range(n)]
        for r in range(R):
            assert outs[r][e] == want


def test_one_data_area_lets_a_rank_overwrite_what_a_peer_still_reads():
    """The model has teeth: with a single data area, a fast rank starts its next call and copies its
    new input over the range a slow peer has yet to sum for the previous call."""
    found = False
    for seed in range(40):
        w, _, _ = simulate(2, 1, 16, 4, False, seed, areas=1, slow={1: 30.0})
        if w.errors:
            found = True
            break
    assert found, "a single data area never showed the overwrite"
    w, _, _ = simulate(2, 1, 16, 4, False, seed, areas=2, slow={1: 30.0})
    assert not w.errors
