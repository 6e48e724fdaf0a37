"""Tile-schedule rule -- TEST INFRASTRUCTURE ONLY (part of the oracle).

The pages' kernel ("Varlen Flash Attention Implementation Plan", Task 1
Step 1) maps a block to (q tile, head) from a global tile start and a linear
scan over cu_seqlens_q; that mapping does not cover every token, so the
schedule here is the plain rule the scheduler kernel must reproduce:

  * one work item per (sequence b, local q tile i, head h) for every
    sequence with Lq_b > 0, where tile i holds local query rows
    [i*BQ, min(Lq_b, (i+1)*BQ));
  * it visits the BK-wide key tiles [first, end) that hold at least one key
    the tile's rows may see, and its cost is end - first.  Without a mask
    first = 0 and end = ceil(Lk_b / BK); with a causal mask end =
    ceil(clamp(min(Lq_b, (i+1)*BQ) + off, 0, Lk_b) / BK), because the tile's
    last row min(Lq_b, (i+1)*BQ) - 1 sees keys up to that row + off (off = 0
    for the top-left mask, Lk_b - Lq_b for the bottom-right one); a sliding
    window of W keys also hides keys below row + off - W, so the tile's first
    row i*BQ gives first = floor(max(0, i*BQ + off - W) / BK).  A tile whose
    rows see no key at all has first = end = 0;
  * the items of one (b, h) form a group and stay next to each other, so
    the q tiles that share a sequence's keys and values run at the same time;
  * groups are ordered by their largest item cost, then their total cost,
    both descending, then by (b, h) ascending (longest work first keeps the
    tail short when CTAs take items in list order);
  * inside a group, tiles are ordered by cost descending, then i ascending;
    with a sliding window by i descending (window costs rise, stay flat,
    then fall, so this is longest first wherever the keys reach past the
    last query, and it keeps a closed form);
  * when the kernel processes two q tiles per work item (`pair`), consecutive
    tiles of a group form one item (the second slot is empty for the last
    tile of a group with an odd count); otherwise each tile is one item.

Each item is eight int32: (b, i_a, h, end_a, i_b, end_b, first_a,
first_b), with i_b = -1 and end_b = first_b = 0 when the second slot is
empty; without a window first_a = first_b = 0 and end is the cost.  Integer work: the
scheduler kernel must match this bit for bit.
"""
from __future__ import annotations

import numpy as np


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def tile_range(lq: int, lk: int, i: int, bq: int, bk: int, causal,
               window_left: int = -1) -> tuple[int, int]:
    """Key tiles [first, end) that q tile i of a (lq, lk) sequence must visit.

    causal: 0 / False no mask, 1 / True top-left, 2 bottom-right;
    window_left >= 0 (with a causal mode) hides keys j < row + off - window_left."""
    if not causal:
        return 0, _ceil_div(lk, bk)
    off = lk - lq if int(causal) == 2 else 0
    # the rows' visible keys form one run [k_lo, k_hi): the last row's
    # diagonal bounds it above, the first row's window edge below
    k_hi = max(0, min(lk, min(lq, (i + 1) * bq) + off))
    k_lo = max(0, i * bq + off - window_left) if window_left >= 0 else 0
    if k_lo >= k_hi:
        return 0, 0
    return k_lo // bk, _ceil_div(k_hi, bk)


def tile_cost(lq: int, lk: int, i: int, bq: int, bk: int, causal, window_left: int = -1) -> int:
    """Number of key tiles that q tile i of a (lq, lk) sequence must visit."""
    first, end = tile_range(lq, lk, i, bq, bk, causal, window_left)
    return end - first


def schedule(cu_seqlens_q, cu_seqlens_k, num_heads: int, bq: int, bk: int,
             causal, pair: bool = False, window_left: int = -1) -> np.ndarray:
    """The ordered work list, int32 [n_items, 8] of
    (b, i_a, h, end_a, i_b, end_b, first_a, first_b)."""
    cq = [int(x) for x in cu_seqlens_q]
    ck = [int(x) for x in cu_seqlens_k]
    groups = []
    for b in range(len(cq) - 1):
        lq = cq[b + 1] - cq[b]
        lk = ck[b + 1] - ck[b]
        tiles = [tile_range(lq, lk, i, bq, bk, causal, window_left) + (i,)
                 for i in range(_ceil_div(lq, bq))]
        if not tiles:
            continue
        if window_left >= 0 and causal:
            tiles.sort(key=lambda t: -t[2])
        else:
            tiles.sort(key=lambda t: (t[0] - t[1], t[2]))
        biggest = max(e - f for f, e, _ in tiles)
        total = sum(e - f for f, e, _ in tiles)
        step = 2 if pair else 1
        for h in range(num_heads):
            members = []
            for k in range(0, len(tiles), step):
                fa, ea, ia = tiles[k]
                fb, eb, ib = tiles[k + 1] if step == 2 and k + 1 < len(tiles) else (0, 0, -1)
                members.append((b, ia, h, ea, ib, eb, fa, fb))
            groups.append(((-biggest, -total, b, h), members))
    groups.sort(key=lambda g: g[0])
    items = [it for _, members in groups for it in members]
    out = np.zeros((len(items), 8), dtype=np.int32)
    for n, it in enumerate(items):
        out[n] = it
    return out
