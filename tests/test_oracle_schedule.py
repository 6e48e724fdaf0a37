"""Pins for the tile-schedule rule (CPU only, integers).

  * brute force: an item's cost equals the number of key tiles holding at
    least one (row, key) pair the mask lets through, found by enumeration;
  * coverage: every (sequence, q tile, head) appears exactly once and the
    tiles cover every query row of every head once;
  * order: the items of one (sequence, head) are contiguous; groups come in
    non-increasing order of their largest cost, then total cost; costs never
    increase inside a group.
"""
import numpy as np
import pytest

from variable_length_flashattention_gb300 import workloads as W


def _brute_cost(lq, lk, i, bq, bk, causal):
    rows = range(i * bq, min(lq, (i + 1) * bq))
    off = lk - lq if causal == 2 else 0          # 2: bottom-right alignment
    n = 0
    for j in range(-(-lk // bk)):
        keys = range(j * bk, min(lk, (j + 1) * bk))
        if any((not causal) or c <= r + off for r in rows for c in keys):
            n += 1
    return n


@pytest.mark.parametrize("causal", [False, True, 2])
@pytest.mark.parametrize("bq,bk", [(128, 128), (128, 64), (64, 128)])
def test_cost_matches_enumeration(oracle_mod, causal, bq, bk):
    rng = np.random.default_rng(0)
    lq = [int(x) for x in rng.integers(0, 400, 12)] + [1, 128, 129, 256, 0, 300]
    lk = [int(x) for x in rng.integers(0, 400, 12)] + [1, 128, 129, 255, 7, 0]
    cq, ck = W.cu_seqlens(lq), W.cu_seqlens(lk)
    for pair in (False, True):
        items = oracle_mod.schedule(cq, ck, 2, bq, bk, causal, pair)
        for b, ia, h, ca, ib, cb, _, _ in items:
            assert ca == _brute_cost(lq[b], lk[b], ia, bq, bk, causal)
            if ib >= 0:
                assert cb == _brute_cost(lq[b], lk[b], ib, bq, bk, causal)
            else:
                assert cb == 0


def _tiles(items):
    """Expand items into (b, i, h, cost) tiles in list order."""
    out = []
    for b, ia, h, ca, ib, cb, _, _ in items:
        out.append((int(b), int(ia), int(h), int(ca)))
        if ib >= 0:
            out.append((int(b), int(ib), int(h), int(cb)))
    return out


@pytest.mark.parametrize("pair", [False, True])
@pytest.mark.parametrize("causal", [False, True, 2])
def test_coverage_and_order(oracle_mod, causal, pair):
    lq, lk = W.cross_lengths(3)
    H = 5
    cq, ck = W.cu_seqlens(lq), W.cu_seqlens(lk)
    items = oracle_mod.schedule(cq, ck, H, 128, 128, causal, pair)
    tiles = _tiles(items)
    seen = set()
    rows = 0
    for b, i, h, c in tiles:
        key = (b, i, h)
        assert key not in seen
        seen.add(key)
        assert 0 <= i * 128 < lq[b]
        rows += min(lq[b], (i + 1) * 128) - i * 128
    assert rows == sum(lq) * H
    assert len(seen) == H * sum(-(-x // 128) for x in lq)
    # groups contiguous, keyed by (largest cost, total cost) non-increasing
    runs = []
    for b, i, h, c in tiles:
        if not runs or runs[-1][0] != (b, h):
            runs.append(((b, h), []))
        runs[-1][1].append((c, i))
    assert len({r[0] for r in runs}) == len(runs), "a group is split"
    keys = [(-max(c for c, _ in m), -sum(c for c, _ in m), g) for g, m in runs]
    assert keys == sorted(keys)
    for _, m in runs:
        assert [(-c, i) for c, i in m] == sorted((-c, i) for c, i in m)
    # pairs: both slots from one group; only a group's last item may be half empty
    for n, (b, ia, h, ca, ib, cb, z0, z1) in enumerate(items):
        assert z0 == 0 and z1 == 0
        if not pair:
            assert ib == -1 and cb == 0
        elif ib < 0:
            assert n + 1 == len(items) or (items[n + 1][0], items[n + 1][2]) != (b, h)


def test_tiny_workload_list():
    import oracle
    items = oracle.schedule(W.cu_seqlens([1, 7, 64, 129]), W.cu_seqlens([1, 7, 64, 129]),
                            2, 128, 128, True)
    # five q tiles (one per short sequence, two for the 129-token one) times two heads
    assert len(items) == 10
    assert [tuple(x[:4]) for x in items[:4]] == [(3, 1, 0, 2), (3, 0, 0, 1), (3, 1, 1, 2), (3, 0, 1, 1)]
    paired = oracle.schedule(W.cu_seqlens([1, 7, 64, 129]), W.cu_seqlens([1, 7, 64, 129]),
                             2, 128, 128, True, pair=True)
    # the 129-token sequence's two tiles share one item per head
    assert len(paired) == 8
    assert tuple(paired[0]) == (3, 1, 0, 2, 0, 1, 0, 0)
