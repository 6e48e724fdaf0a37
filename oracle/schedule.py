"""Tile-schedule rule -- TEST INFRASTRUCTURE ONLY (part of the oracle).

The pages' kernel ("Varlen Flash Attention Implementation Plan", Task 1
Step 1) maps a block to (q tile, head) from a global tile start and a linear
scan over cu_seqlens_q; that mapping does not cover every token, so the
schedule here is the plain rule the scheduler kernel must reproduce:

  * one work item per (sequence b, local q tile i, head h) for every
    sequence with Lq_b > 0, where tile i holds local query rows
    [i*BQ, min(Lq_b, (i+1)*BQ));
  * its cost is the number of BK-wide key tiles that hold at least one key
    the tile's rows may see: ceil(Lk_b / BK) without a mask, and with a
    causal mask ceil(clamp(min(Lq_b, (i+1)*BQ) + off, 0, Lk_b) / BK), because
    the tile's last row min(Lq_b, (i+1)*BQ) - 1 sees keys 0 .. that row + off
    (off = 0 for the top-left mask, Lk_b - Lq_b for the bottom-right one);
  * the items of one (b, h) form a group and stay next to each other, so
    the q tiles that share a sequence's keys and values run at the same time;
  * groups are ordered by their largest item cost, then their total cost,
    both descending, then by (b, h) ascending (longest work first keeps the
    tail short when CTAs take items in list order);
  * inside a group, tiles are ordered by cost descending, then i ascending;
  * when the kernel processes two q tiles per work item (`pair`), consecutive
    tiles of a group form one item (the second slot is empty for the last
    tile of a group with an odd count); otherwise each tile is one item.

Each item is eight int32: (b, i_a, h, cost_a, i_b, cost_b, 0, 0), with
i_b = -1 and cost_b = 0 when the second slot is empty.  Integer work: the
scheduler kernel must match this bit for bit.
"""
from __future__ import annotations

import numpy as np


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def tile_cost(lq: int, lk: int, i: int, bq: int, bk: int, causal) -> int:
    """Number of key tiles that q tile i of a (lq, lk) sequence must visit.

    causal: 0 / False no mask, 1 / True top-left, 2 bottom-right."""
    if not causal:
        return _ceil_div(lk, bk)
    off = lk - lq if int(causal) == 2 else 0
    last_row_plus_one = min(lq, (i + 1) * bq)
    return _ceil_div(max(0, min(lk, last_row_plus_one + off)), bk)


def schedule(cu_seqlens_q, cu_seqlens_k, num_heads: int, bq: int, bk: int,
             causal, pair: bool = False) -> np.ndarray:
    """The ordered work list, int32 [n_items, 8] of (b, i_a, h, cost_a, i_b, cost_b, 0, 0)."""
    cq = [int(x) for x in cu_seqlens_q]
    ck = [int(x) for x in cu_seqlens_k]
    groups = []
    for b in range(len(cq) - 1):
        lq = cq[b + 1] - cq[b]
        lk = ck[b + 1] - ck[b]
        tiles = [(tile_cost(lq, lk, i, bq, bk, causal), i) for i in range(_ceil_div(lq, bq))]
        if not tiles:
            continue
        tiles.sort(key=lambda t: (-t[0], t[1]))
        biggest = max(c for c, _ in tiles)
        total = sum(c for c, _ in tiles)
        step = 2 if pair else 1
        for h in range(num_heads):
            members = []
            for k in range(0, len(tiles), step):
                ca, ia = tiles[k]
                cb, ib = tiles[k + 1] if step == 2 and k + 1 < len(tiles) else (0, -1)
                members.append((b, ia, h, ca, ib, cb, 0, 0))
            groups.append(((-biggest, -total, b, h), members))
    groups.sort(key=lambda g: g[0])
    items = [it for _, members in groups for it in members]
    out = np.zeros((len(items), 8), dtype=np.int32)
    for n, it in enumerate(items):
        out[n] = it
    return out
