"""The AUTO table (csrc/ar_auto_table.h) and the tool that writes it (tune.py), checked on the CPU.

- `tune.table` keeps the fastest measurement per (element size, R, row length, tokens), turns the
  measured token counts into ascending ranges, leaves the last range open, and ends with the sentinel.
- Every committed entry is well formed, and the ranges of one row shape ascend to an open end.
- Every committed entry is what AUTO launches over its whole token range: ar_query_launch reports
  the entry's strategy, kernel, units per thread, residual_out order, cluster size or blocks per SM,
  and stage cap.  So no entry quietly falls back to the rule because its shape does not fit.
"""
import ctypes
import json
import re
import shutil

import pytest

import tensor_allreduce_residual_gb300 as ar
from tensor_allreduce_residual_gb300 import _build, tune

ENTRY = re.compile(r"^\s*\{(\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+)\},")
INT_MAX = 2 ** 31 - 1
KERNEL_OF_MODE = {0: 1, 1: 2, 2: 3, 3: 4, 4: 6}   # OneShotMode -> ar_kernel


def entries(text):
    return [tuple(int(x) for x in m.groups()) for m in map(ENTRY.match, text.splitlines()) if m]


def committed():
    rows = entries(open(tune.TABLE).read())
    assert rows and rows[-1] == (0,) * 10, "the table ends with its sentinel"
    return rows[:-1]


@pytest.fixture(scope="module")
def L():
    _build.build()
    return ar.lib()


def test_table_from_a_sweep(tmp_path, monkeypatch):
    table = tmp_path / "ar_auto_table.h"
    shutil.copy(tune.TABLE, table)
    monkeypatch.setattr(tune, "TABLE", str(table))
    shape = dict(case="c", esize=2, R=8, units_row=1024)
    recs = [
        dict(shape, T=1, strategy="ONESHOT", shape="1:4:0:8", us=3.1),
        dict(shape, T=1, strategy="ONESHOT", shape="2:0:1", us=4.0),
        dict(shape, T=1, strategy="TWOSHOT", shape="-", us=4.4),
        dict(shape, T=64, strategy="TWOSHOT", shape="-", us=3.0),
        dict(shape, T=64, strategy="ONESHOT", shape="2:0:1", us=3.9),
        dict(shape, T=8192, strategy="ONESHOT", shape="2:3:1:1:2", us=207.0),
        dict(shape, T=8192, strategy="ONESHOT", shape="4:1:0", us=231.5),
    ]
    sweep = tmp_path / "sweep.jsonl"
    sweep.write_text("".join(json.dumps(r) + "\n" for r in recs))
    tune.table(str(sweep))
    assert entries(table.read_text()) == [
        (2, 8, 1024, 1, 1, 1, 4, 0, 8, 0),          # fastest at one token: the 8-block cluster shape
        (2, 8, 1024, 64, 2, 0, 0, 0, 1, 0),         # two-shot won at 64 tokens
        (2, 8, 1024, INT_MAX, 1, 2, 3, 1, 1, 2),    # the last range is open
        (0,) * 10]
    assert "8192: one-shot 207.0 us" in table.read_text()


def test_committed_entries_are_well_formed_and_ordered():
    ranges = {}
    for esize, R, units, tmax, strategy, vpt, mode, early, bps, stages in committed():
        assert esize in (2, 4) and 1 <= R <= ar.AR_MAX_RANKS and units > 0 and tmax > 0
        assert strategy in (ar.AR_ONESHOT, ar.AR_TWOSHOT)
        if strategy == ar.AR_ONESHOT:
            assert vpt in (1, 2, 4, 8) and mode in KERNEL_OF_MODE and early in (0, 1)
            assert bps >= 1 and 0 <= stages <= 16
        ranges.setdefault((esize, R, units), []).append(tmax)
    for key, tmaxes in ranges.items():
        assert tmaxes == sorted(set(tmaxes)), key
        assert tmaxes[-1] == INT_MAX, key


def test_committed_entries_are_what_auto_launches(L):
    low = {}
    for e in committed():
        esize, R, units, tmax, strategy, vpt, mode, early, bps, stages = e
        hidden = units * (16 // esize)
        first = low.get((esize, R, units), 0) + 1
        low[(esize, R, units)] = tmax
        last = tmax if tmax < INT_MAX else max(first, 8192)
        for T in sorted({first, (first + last) // 2, last}):
            for dt in ((ar.AR_FP16, ar.AR_BF16) if esize == 2 else (ar.AR_FP32,)):
                plan = ar.ArLaunchPlan()
                assert L.ar_query_launch(R, hidden, T, dt, ar.AR_AUTO, ctypes.byref(plan)) == ar.AR_OK
                where = (e, T, dt)
                assert plan.strategy == strategy, where
                if strategy == ar.AR_TWOSHOT:
                    assert plan.kernel == 5, where
                    continue
                want = KERNEL_OF_MODE[mode]
                if mode == 2:   # the persistent kernel needs whole-warp rows and R in {1, 2, 4, 8}
                    want = (2, 3)
                assert plan.kernel in (want if isinstance(want, tuple) else (want,)), where
                assert plan.units_per_thread == vpt, where
                assert plan.early_residual == early, where
                if mode == 4:
                    assert plan.cluster == bps, where
                if mode == 3:
                    assert plan.blocks_per_sm == bps, where
                    assert stages == 0 or plan.stages <= stages, where


def test_sweep_skips_a_shape_that_does_not_fit():
    """tune.shape_taken: a plan that is not the shape asked for (the rule's fallback) is not recorded
    under that shape's name.  Plans here are written out by hand."""
    base = dict(strategy=1, kernel=4, units_per_thread=2, early_residual=1, cluster=0, blocks_per_sm=1, stages=2)
    assert tune.shape_taken(base, "2:3:1:1:2")
    assert tune.shape_taken(base, "2:3:1:1")                         # no stage cap asked for
    assert not tune.shape_taken(dict(base, stages=4), "2:3:1:1:2")  # more stages than the cap
    assert not tune.shape_taken(dict(base, kernel=1, units_per_thread=4), "1:3:1:1:8")  # fell back to the rule
    assert not tune.shape_taken(dict(base, early_residual=0), "2:3:1")
    cluster = dict(base, kernel=6, units_per_thread=1, early_residual=0, cluster=8, blocks_per_sm=0, stages=0)
    assert tune.shape_taken(cluster, "1:4:0:8") and not tune.shape_taken(cluster, "1:4:0:4")
    staged = dict(base, kernel=2, units_per_thread=4, early_residual=0, blocks_per_sm=0, stages=0)
    assert tune.shape_taken(staged, "4:1:0") and tune.shape_taken(staged, "4:2:0")   # persistent -> staged
    assert not tune.shape_taken(dict(staged, strategy=2, kernel=5), "4:1:0")


SUM_ENTRY = re.compile(r"^\s*\{(\d+), (\d+), (\d+)LL, (\d+)\},")
LLONG_MAX = 2 ** 63 - 1


def sum_entries(text):
    return [tuple(int(x) for x in m.groups()) for m in map(SUM_ENTRY.match, text.splitlines()) if m]


def test_sum_table_from_a_sweep(tmp_path, monkeypatch):
    """The faster partition per measured n, rank slices only beyond the noise margin, merged into ranges."""
    table = tmp_path / "ar_auto_table.h"
    shutil.copy(tune.TABLE, table)
    monkeypatch.setattr(tune, "TABLE", str(table))
    recs = []
    for units, one, two in [(64, 1.70, 1.60), (128, 1.80, 1.62), (256, 2.00, 1.99), (512, 2.20, 2.30),
                            (1024, 3.00, 2.50), (2048, 5.0, 5.2)]:
        recs += [dict(R=4, esize=2, n=units * 8, units=units, strategy="ONESHOT", us=one),
                 dict(R=4, esize=2, n=units * 8, units=units, strategy="TWOSHOT", us=two)]
    sweep = tmp_path / "sums.jsonl"
    sweep.write_text("".join(json.dumps(r) + "\n" for r in recs))
    tune.sum_table(str(sweep))
    assert sum_entries(table.read_text()) == [
        (2, 4, 128, 2),        # rank slices clearly faster up to 128 vectors
        (2, 4, 512, 1),        # within 2 % at 256 (one slice kept), slower at 512
        (2, 4, 1024, 2),
        (2, 4, LLONG_MAX, 1),  # the last range is open
    ]
    # the fused table is untouched
    assert entries(table.read_text()) == entries(open(tune.TABLE).read())


def test_reduce_only_auto_is_the_table_choice(L):
    """ar_query_strategy(..., AR_FUSION_NONE) reports, at every measured size of every committed entry
    range, the partition the table names (AUTO in ar_sum takes the same function)."""
    rows = sum_entries(open(tune.TABLE).read())
    for esize, R, umax, strategy in rows:
        dtype = ar.AR_FP16 if esize == 2 else ar.AR_FP32
        lanes = 16 // esize
        lo = max([u for e, r, u, _ in rows if e == esize and r == R and u < umax], default=0)
        for units in {lo + 1, min(umax, 1 << 26)}:
            s, _ = ar.ar_query_strategy(R, units * lanes, 0, dtype, ar.AR_FUSION_NONE)
            assert s == strategy, (esize, R, units, s, strategy)
