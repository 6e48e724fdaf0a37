"""Work accounting for throughput figures (not part of the computed result).

Algorithmic FLOPs of the varlen forward count only the (query, key) pairs the
mask lets through: 4 * H * D per pair (2 for the q.k product, 2 for p * v).
Masked or padded tile work and the exp / max / sum work are not counted.
Algorithmic bytes of a decode pass count every K/V byte of the listed blocks
once, plus q, the fp32 state read and written by each step, and the output.
"""
from __future__ import annotations


def attended_pairs(lengths_q, lengths_k, causal: bool) -> int:
    """Pairs per head; causal is top-left: local key j visible to local query i iff j <= i."""
    total = 0
    for lq, lk in zip(lengths_q, lengths_k):
        lq, lk = int(lq), int(lk)
        if not causal:
            total += lq * lk
        else:
            r = min(lq, lk)          # rows i < r see i + 1 keys; rows i >= lk see all lk keys
            total += r * (r + 1) // 2 + (lq - r) * lk
    return total


def varlen_flops(case) -> int:
    return 4 * case.num_heads * case.head_dim * attended_pairs(case.lengths_q, case.lengths_k,
                                                              case.causal)


def varlen_bwd_flops(case) -> int:
    """Backward: five products per attended pair (S = q.k, dP = dout.v, dV += P dout,
    dK += dS q, dQ += dS k), 2 * D each, so 10 * H * D per pair (2.5 x the forward)."""
    return 10 * case.num_heads * case.head_dim * attended_pairs(case.lengths_q, case.lengths_k,
                                                               case.causal)


def varlen_context_bytes(case) -> int:
    """Bytes read (q, k, v bf16) and written (out bf16, lse f32) once each."""
    H, D = case.num_heads, case.head_dim
    return 2 * (case.total_q + 2 * case.total_k) * H * D + (2 * D + 4) * case.total_q * H


def decode_step_active(case, t: int) -> int:
    cap = case.tile_capacity
    return sum(1 for n in case.n_blocks if n > t * cap)


def decode_bytes(case) -> int:
    """One full decode pass: init + every step + finalize."""
    S, Hq, D = case.num_seqs, case.num_q_heads, case.head_dim
    state = S * Hq * (D + 2) * 4
    total = state                                   # init writes the state
    for t in range(case.num_steps):
        active = decode_step_active(case, t)
        total += active * Hq * D * 2                 # q of the active sequences
        total += 2 * active * Hq * (D + 2) * 4       # state read + written
        total += active * (case.tile_capacity + 1) * 4  # block ids and count
    total += case.kv_bytes()
    total += state + S * Hq * D * 2                 # finalize reads l, o, writes bf16 out
    return total
