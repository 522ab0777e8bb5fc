"""A CPU model of the Lamport-style kernel's schedule, checked before trusting it on a GPU.

The kernel deals its groups (rows, or row slices when a row is split over
C blocks) out in steps of the grid G: in a step, block b pushes the group at
position b and then reduces the group at position (b + 1) mod G; a position
that a short last step does not reach is skipped.  With separate push and
reduce warps (rows not split), a block's pushes run through the steps on
their own and its reduces on their own: two chains of program order.  A split row's blocks
exchange their shares of the sum of squares and wait for all C of them.  The
buffer is a ring of D steps (2 by default): group g lives in ring slot g mod DG, and a
block pushing a group into a slot that held an earlier group of the call
first waits for the block that reduced that earlier group to publish the
step in which it did so.  Blocks wait on one another, so the schedule must
(1) push and reduce every group exactly once, (2) keep every split row's
slices in one step, (3) have no cycle among its waits, whatever the grid,
(4) give every ring slot the same reducer in every step (so a reducer never
mistakes the slot's previous contents for new data: it wrote the marker
there itself), and (5) make every push into a reused slot wait for the
reduce of the slot's previous group.  This model states those rules
independently of the CUDA code and checks them for many token counts,
splits and grids, including a grid rounded down to whole split rows as the
launcher does.
"""
import random
from collections import defaultdict, deque

import pytest


def schedule(groups, G):
    """[(step, block, pushed group or None, reduced group or None)] for every block in every step."""
    out = []
    step = 0
    for base in range(0, groups, G):
        n = min(G, groups - base)
        for b in range(G):
            q = (b + 1) % G
            out.append((step, b, base + b if b < n else None, base + q if q < n else None))
        step += 1
    return out


def schedule_short_step_wraps(groups, G):
    """The earlier mapping: in a short last step of n groups, block b reduced position (b + 1) mod n."""
    out = []
    step = 0
    for base in range(0, groups, G):
        n = min(G, groups - base)
        for b in range(n):
            out.append((step, b, base + b, base + (b + 1) % n))
        step += 1
    return out


def check(tokens, csize, rows, G, launcher_grid=True, roles=False, ring_steps=2):
    groups = tokens * csize if csize > 1 else -(-tokens // rows)
    sched = schedule(groups, G)
    pushed = [g for _, _, g, _ in sched if g is not None]
    reduced = [g for _, _, _, g in sched if g is not None]
    assert sorted(pushed) == list(range(groups))
    assert sorted(reduced) == list(range(groups))
    step_of = {g: s for s, _, g, _ in sched if g is not None}
    if csize > 1 and launcher_grid:   # the launcher's grid: all slices of a row are reduced in one step
        assert G % csize == 0
        for row in range(tokens):
            assert len({step_of[row * csize + c] for c in range(csize)}) == 1

    ring = ring_steps * G                                 # ring slots, in groups
    pusher = {g: (s, b) for s, b, g, _ in sched if g is not None}
    reducer = {g: (s, b) for s, b, _, g in sched if g is not None}
    for g in range(ring, groups):                         # (4) one reducer block per ring slot
        assert reducer[g][1] == reducer[g - ring][1], (g, reducer[g], reducer[g - ring])

    # Wait graph.  Nodes: ("push", s, b), ("share", s, b) = its reduce has read its data and written
    # its share, ("done", s, b) = its step is complete (published).  Edges point from what must happen
    # first.
    edges = defaultdict(set)
    nodes = set()
    for s, b, gp, gr in sched:
        nodes |= {("push", s, b), ("share", s, b), ("done", s, b)}
        edges[("push", s, b)].add(("share", s, b))              # program order within a step
        edges[("share", s, b)].add(("done", s, b))
        if gr is not None:
            ps, pb = pusher[gr]
            edges[("push", ps, pb)].add(("share", s, b))        # the reduce polls the pushed group
        if gp is not None and gp >= ring:                       # (5) a reused slot: the progress wait
            ws, wb = s - ring_steps, (b + G - 1) % G            # what the kernel waits for ...
            assert reducer[gp - ring] == (ws, wb)               # ... is the reduce of the slot's last group
            edges[("done", ws, wb)].add(("push", s, b))
    steps = max(s for s, _, _, _ in sched) + 1
    for b in range(G):                                          # program order across steps
        for s0 in range(steps - 1):
            if roles:   # separate push and reduce warps: two chains per block
                edges[("push", s0, b)].add(("push", s0 + 1, b))
                edges[("done", s0, b)].add(("share", s0 + 1, b))
            else:
                edges[("done", s0, b)].add(("push", s0 + 1, b))
        if roles:       # within a step the reduce no longer follows the block's own push
            for s0 in range(steps):
                edges[("push", s0, b)].discard(("share", s0, b))
    if csize > 1:                                               # a split row's exchange waits for every share
        for row in range(tokens):
            members = [reducer[row * csize + c] for c in range(csize)]
            for (s0, b0) in members:
                for (s1, b1) in members:
                    edges[("share", s0, b0)].add(("done", s1, b1))
    # Kahn's algorithm: every node must come out, or the waits contain a cycle.
    indeg = {v: 0 for v in nodes}
    for u in edges:
        for v in edges[u]:
            indeg[v] += 1
    ready = deque(v for v in nodes if indeg[v] == 0)
    seen = 0
    while ready:
        u = ready.popleft()
        seen += 1
        for v in edges.get(u, ()):
            indeg[v] -= 1
            if indeg[v] == 0:
                ready.append(v)
    assert seen == len(nodes), f"waits form a cycle: tokens={tokens} csize={csize} rows={rows} G={G}"


@pytest.mark.parametrize("csize", [1, 2, 4, 8])
def test_schedule_covers_every_group_once_without_cycles(csize):
    rng = random.Random(csize)
    for _ in range(150):
        tokens = rng.choice([1, 2, 3, 7, 8, 16, 33, 100, 257, rng.randint(1, 700)])
        rows = 1 if csize > 1 else rng.choice([1, 2, 4, 8])
        groups = tokens * csize if csize > 1 else -(-tokens // rows)
        resident = rng.choice([1, 2, 5, 152, 304, 456, rng.randint(1, 1000)])
        cap = resident // csize * csize               # the launcher's rounding to whole split rows
        if cap < csize:
            continue
        check(tokens, csize, rows, min(groups, cap))


def test_grid_not_a_multiple_of_the_split_would_straddle_steps():
    """Why the launcher rounds the grid down to whole split rows: with 6 blocks and rows split over 4,
    the second row's slices fall into two steps."""
    groups, G, csize = 8, 6, 4
    step_of = {gr: s for s, _, _, gr in schedule(groups, G) if gr is not None}
    assert len({step_of[4 + c] for c in range(csize)}) == 2


def test_the_model_finds_the_cycle_of_a_straddling_row():
    """The model has teeth: one row split over 4 blocks on a grid of 3 (which the launcher never
    makes).  Block 0 reduces slice 1 in step 0 and slice 3 in step 1, so its exchange in step 0 waits
    for a share it would only write after leaving step 0: a cycle."""
    with pytest.raises(AssertionError, match="cycle"):
        check(1, 4, 1, 3, launcher_grid=False)
    check(1, 4, 1, 4)   # the launcher's grid for this call


def test_a_short_last_step_must_not_change_a_ring_slot_reducer():
    """Why a short last step skips positions instead of wrapping at n: with 5 groups on a grid of 2 the
    ring of 4 slots is reused by group 4, and reducing (b + 1) mod n in the last step (n = 1) gives
    slot 0 a reducer other than the block that emptied it two steps before.  That block could still
    be about to write the marker back when the new reducer reads the slot, and take the old group's
    data for the new group's."""
    G, groups = 2, 5
    old = {g: b for _, b, _, g in schedule_short_step_wraps(groups, G)}
    new = {g: b for _, b, _, g in schedule(groups, G) if g is not None}
    assert old[4] != old[0]
    assert new[4] == new[0]
    check(5, 1, 1, 2)


@pytest.mark.parametrize("tokens,G", [(8192, 304), (3000, 512), (2500, 152), (20000 // 8, 512)])
def test_prefill_sized_rings(tokens, G):
    """Shapes of the GPU tests whose rows outnumber the ring: every slot reused several times."""
    check(tokens, 1, 1, G)


def test_separate_push_and_reduce_warps_cover_every_group_without_cycles():
    """The same rules when a block's push warps and reduce warps run apart (rows not split): pushes
    ahead of their own block's reduces, limited only by the ring's progress waits."""
    rng = random.Random(99)
    for _ in range(200):
        tokens = rng.choice([1, 2, 7, 33, 257, 1000, rng.randint(1, 5000)])
        rows = rng.choice([1, 2, 4])
        groups = -(-tokens // rows)
        G = min(groups, rng.choice([1, 2, 5, 152, 304, 512, rng.randint(1, 512)]))
        check(tokens, 1, rows, G, roles=True)


@pytest.mark.parametrize("ring_steps", [3, 4])
def test_deeper_rings(ring_steps):
    rng = random.Random(ring_steps)
    for _ in range(100):
        tokens = rng.choice([1, 33, 700, 3000, rng.randint(1, 6000)])
        rows = rng.choice([1, 2, 4])
        groups = -(-tokens // rows)
        G = min(groups, 1024 // ring_steps, rng.choice([1, 5, 152, 256, rng.randint(1, 341)]))
        check(tokens, 1, rows, G, roles=rng.random() < 0.5, ring_steps=ring_steps)
