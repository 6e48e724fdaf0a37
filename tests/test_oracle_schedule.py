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


def _visible_tiles(lq, lk, i, bq, bk, causal, window_left=-1):
    """Key tiles holding at least one (row, key) pair the mask lets through."""
    rows = range(i * bq, min(lq, (i + 1) * bq))
    off = lk - lq if causal == 2 else 0          # 2: bottom-right alignment
    seen = []
    for j in range(-(-lk // bk)):
        keys = range(j * bk, min(lk, (j + 1) * bk))
        if any((not causal) or (c <= r + off and (window_left < 0 or c >= r + off - window_left))
               for r in rows for c in keys):
            seen.append(j)
    return seen


def _brute_cost(lq, lk, i, bq, bk, causal):
    return len(_visible_tiles(lq, lk, i, bq, bk, causal))


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


@pytest.mark.parametrize("causal", [1, 2])
@pytest.mark.parametrize("window_left", [0, 1, 63, 64, 127, 200, 1000])
@pytest.mark.parametrize("bq,bk", [(128, 128), (128, 64)])
def test_window_range_matches_enumeration(oracle_mod, causal, window_left, bq, bk):
    # [first, end) is exactly the run of key tiles with a visible pair: the
    # visible tiles are contiguous, so the range visits no empty tile
    rng = np.random.default_rng(window_left)
    lq = [int(x) for x in rng.integers(0, 700, 10)] + [1, 128, 129, 600, 0, 300]
    lk = [int(x) for x in rng.integers(0, 700, 10)] + [1, 128, 129, 250, 7, 0]
    cq, ck = W.cu_seqlens(lq), W.cu_seqlens(lk)
    for pair in (False, True):
        items = oracle_mod.schedule(cq, ck, 2, bq, bk, causal, pair, window_left=window_left)
        for b, ia, h, ea, ib, eb, fa, fb in items:
            for i, f, e in ((ia, fa, ea), (ib, fb, eb)):
                if i < 0:
                    assert (f, e) == (0, 0)
                    continue
                vis = _visible_tiles(lq[b], lk[b], i, bq, bk, causal, window_left)
                assert (f, e) == ((vis[0], vis[-1] + 1) if vis else (0, 0))
                assert vis == list(range(f, e))
            if pair and ib >= 0 and ea > fa and eb > fb:
                # the two slots' ranges touch or overlap: their union is one run
                assert max(fa, fb) <= min(ea, eb)


@pytest.mark.parametrize("pair", [False, True])
def test_window_coverage_and_order(oracle_mod, pair):
    lq, lk = W.cross_lengths(3)
    H = 3
    cq, ck = W.cu_seqlens(lq), W.cu_seqlens(lk)
    items = oracle_mod.schedule(cq, ck, H, 128, 128, 2, pair, window_left=300)
    tiles = []
    for b, ia, h, ea, ib, eb, fa, fb in items:
        tiles.append((int(b), int(ia), int(h), int(ea - fa)))
        if ib >= 0:
            tiles.append((int(b), int(ib), int(h), int(eb - fb)))
    assert len(set((b, i, h) for b, i, h, _ in tiles)) == len(tiles)
    assert len(tiles) == H * sum(-(-x // 128) for x in lq)
    runs = []
    for b, i, h, c in tiles:
        if not runs or runs[-1][0] != (b, h):
            runs.append(((b, h), []))
        runs[-1][1].append((c, i))
    assert len({r[0] for r in runs}) == len(runs), "a group is split"
    keys = [(-max(c for c, _ in m), -sum(c for c, _ in m), g) for g, m in runs]
    assert keys == sorted(keys)
    for _, m in runs:
        assert [i for _, i in m] == sorted((i for _, i in m), reverse=True)


def test_window_tiny_list():
    import oracle
    # one 300-token causal sequence, window 100: tile 2 (rows 256..299) sees
    # keys 156..299 (tiles 1, 2), tile 1 keys 28..255 (0, 1), tile 0 keys 0..127
    items = oracle.schedule(W.cu_seqlens([300]), W.cu_seqlens([300]), 1, 128, 128, 1,
                            window_left=100)
    assert [tuple(x) for x in items] == [(0, 2, 0, 3, -1, 0, 1, 0), (0, 1, 0, 2, -1, 0, 0, 0),
                                         (0, 0, 0, 1, -1, 0, 0, 0)]
