"""Pins for the paged GQA decode oracle (CPU only).

  * tile fragmentation: one tile of every block, tiles of 32, tiles of 1 and
    an uneven split all give the same final output (the property
    attention_ref.rs states it exists to check);
  * reduction to the varlen forward: decode of (sequence s, q head qh) is
    non-causal varlen attention of one query over the gathered tokens of kv
    head qh / group, scale 1/sqrt(D);
  * a numpy brute force that walks the block table token by token;
  * closed forms: no blocks ever gives m = -inf, l = 0, out = 0; one block
    whose keys are all equal gives the mean of its V rows;
  * the extension for contexts that end inside a block and an explicit scale
    (per-step token counts): a numpy brute force over the first ctx tokens of
    each sequence in block-table order, with that scale; full token counts
    reproduce the default bit for bit.
"""
import math

import numpy as np
import pytest
import torch

from variable_length_flashattention_gb300 import workloads as W


def _small(seed=0, n_blocks=(3, 1, 7, 0, 5), Hq=8, Hkv=2, D=16, bs=4, cap=2):
    rng = np.random.default_rng(seed)
    perm = rng.permutation(sum(n_blocks)).astype(np.int32)
    return W.make_decode("small", list(n_blocks), Hq, Hkv, D, bs, cap, perm, value_seed=seed)


def _run(oracle_mod, case, cap=None):
    """All steps with tiles of `cap` blocks (default: the case's own capacity)."""
    st = oracle_mod.DecodeState(case.num_seqs, case.num_q_heads, case.head_dim)
    cap = cap or case.tile_capacity
    c2 = W.DecodeCase(case.name, case.context_lengths, case.n_blocks, case.num_q_heads,
                      case.num_kv_heads, case.head_dim, case.block_size, cap, case.q,
                      case.k_pool, case.v_pool, case.block_table)
    for t in range(c2.num_steps):
        tb, tc = c2.tile(t)
        oracle_mod.decode_step(st, case.q, case.k_pool, case.v_pool, tb, tc,
                               case.num_kv_heads, case.block_size)
    return st, oracle_mod.decode_finalize(st)


def _brute(case):
    q = case.q.double().numpy()
    K = case.k_pool.double().numpy()
    V = case.v_pool.double().numpy()
    g = case.num_q_heads // case.num_kv_heads
    out = np.zeros((case.num_seqs, case.num_q_heads, case.head_dim))
    for s in range(case.num_seqs):
        for qh in range(case.num_q_heads):
            kh = qh // g
            ks, vs = [], []
            for blk in case.block_table[s]:
                for t in range(case.block_size):
                    ks.append(K[blk, t, kh])
                    vs.append(V[blk, t, kh])
            if not ks:
                continue
            x = np.array(ks) @ q[s, qh] / math.sqrt(case.head_dim)
            w = np.exp(x - x.max())
            out[s, qh] = (w[:, None] * np.array(vs)).sum(0) / w.sum()
    return out


def test_tile_fragmentation_invariance(oracle_mod):
    case = _small(seed=1)
    big = max(case.n_blocks)
    ref_st, ref = _run(oracle_mod, case, cap=big)        # one tile holds every block
    for cap in (1, 2, 3, 32):
        st, out = _run(oracle_mod, case, cap=cap)
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)
        # the state itself: m + ln l is independent of the split
        live = ref_st.l > 0
        np.testing.assert_allclose((st.m + np.log(np.where(st.l > 0, st.l, 1)))[live],
                                   (ref_st.m + np.log(np.where(live, ref_st.l, 1)))[live],
                                   rtol=1e-13, atol=1e-13)


def test_matches_brute_force(oracle_mod):
    case = _small(seed=2)
    _, out = _run(oracle_mod, case)
    np.testing.assert_allclose(out, _brute(case), rtol=1e-11, atol=1e-13)


def test_reduces_to_varlen_single_query(oracle_mod):
    case = _small(seed=3, n_blocks=(2, 4, 1))
    _, out = _run(oracle_mod, case)
    g = case.num_q_heads // case.num_kv_heads
    D = case.head_dim
    for s in range(case.num_seqs):
        for qh in range(case.num_q_heads):
            kh = qh // g
            blocks = case.block_table[s]
            kk = case.k_pool[blocks, :, kh, :].reshape(-1, 1, D).contiguous()
            vv = case.v_pool[blocks, :, kh, :].reshape(-1, 1, D).contiguous()
            qq = case.q[s, qh].reshape(1, 1, D).contiguous()
            cq = np.array([0, 1], np.int32)
            ck = np.array([0, kk.shape[0]], np.int32)
            ref, _, _ = oracle_mod.varlen_fwd(qq, kk, vv, cq, ck, 1, D, 1.0 / math.sqrt(D), False)
            np.testing.assert_allclose(out[s, qh], ref[0, 0], rtol=1e-12, atol=1e-14)


def test_no_blocks_gives_zero(oracle_mod):
    case = _small(seed=4, n_blocks=(0, 3, 0))
    st, out = _run(oracle_mod, case)
    for s in (0, 2):
        assert np.all(out[s] == 0.0)
        assert np.all(st.l[s] == 0.0)
        assert np.all(np.isneginf(st.m[s]))
    assert np.all(st.l[1] > 0)


def test_equal_keys_give_mean_of_block_v(oracle_mod):
    case = _small(seed=5, n_blocks=(1,), cap=1)
    k = case.k_pool.clone()
    k[:] = k[0, 0]                     # every token of the block has the same key row
    case = W.DecodeCase(case.name, case.context_lengths, case.n_blocks, case.num_q_heads,
                        case.num_kv_heads, case.head_dim, case.block_size, 1, case.q, k,
                        case.v_pool, case.block_table)
    _, out = _run(oracle_mod, case)
    v = case.v_pool.double().numpy()
    g = case.num_q_heads // case.num_kv_heads
    for qh in range(case.num_q_heads):
        np.testing.assert_allclose(out[0, qh], v[0, :, qh // g].mean(0), rtol=1e-13, atol=1e-15)


def test_rejects_out_of_range_block_and_count(oracle_mod):
    case = _small(seed=6, n_blocks=(2, 2))
    st = oracle_mod.DecodeState(2, case.num_q_heads, case.head_dim)
    tb, tc = case.tile(0)
    bad = tb.copy()
    bad[1, 0] = case.num_blocks
    with pytest.raises(ValueError):
        oracle_mod.decode_step(st, case.q, case.k_pool, case.v_pool, bad, tc,
                               case.num_kv_heads, case.block_size)
    badc = tc.copy()
    badc[0] = tb.shape[1] + 1
    with pytest.raises(ValueError):
        oracle_mod.decode_step(st, case.q, case.k_pool, case.v_pool, tb, badc,
                               case.num_kv_heads, case.block_size)
    assert np.all(np.isneginf(st.m)) and np.all(st.l == 0)   # nothing was changed


def _brute_exact(case, scale):
    q = case.q.double().numpy()
    K = case.k_pool.double().numpy()
    V = case.v_pool.double().numpy()
    g = case.num_q_heads // case.num_kv_heads
    out = np.zeros((case.num_seqs, case.num_q_heads, case.head_dim))
    lse = np.full((case.num_seqs, case.num_q_heads), -np.inf)
    for s in range(case.num_seqs):
        toks = [(blk, t) for blk in case.block_table[s] for t in range(case.block_size)]
        toks = toks[:case.context_lengths[s]]
        if not toks:
            continue
        for qh in range(case.num_q_heads):
            kh = qh // g
            ks = np.array([K[b, t, kh] for b, t in toks])
            vs = np.array([V[b, t, kh] for b, t in toks])
            x = scale * (ks @ q[s, qh])
            w = np.exp(x - x.max())
            out[s, qh] = (w[:, None] * vs).sum(0) / w.sum()
            lse[s, qh] = x.max() + math.log(w.sum())
    return out, lse


def _run_exact(oracle_mod, case, scale):
    st = oracle_mod.DecodeState(case.num_seqs, case.num_q_heads, case.head_dim)
    for t in range(case.num_steps):
        tb, tc = case.tile(t)
        oracle_mod.decode_step(st, case.q, case.k_pool, case.v_pool, tb, tc, case.num_kv_heads,
                               case.block_size, tile_token_counts=case.tile_tokens(t),
                               scale=scale)
    return st, oracle_mod.decode_finalize(st)


@pytest.mark.parametrize("scale", [0.0, 0.37])
def test_exact_context_and_scale_match_brute_force(oracle_mod, scale):
    n_blocks = (3, 1, 7, 2, 5, 1)
    ctx = [9, 1, 27, 8, 17, 0]          # partial last blocks, a one-token and an empty context
    rng = np.random.default_rng(7)
    perm = rng.permutation(sum(n_blocks)).astype(np.int32)
    case = W.make_decode("exact", list(n_blocks), 8, 2, 16, 4, 2, perm, value_seed=7,
                         context_lengths=ctx)
    eff = scale if scale > 0 else 1.0 / math.sqrt(case.head_dim)
    st, out = _run_exact(oracle_mod, case, scale)
    ref, ref_lse = _brute_exact(case, eff)
    np.testing.assert_allclose(out, ref, atol=1e-12, rtol=0)
    live = np.isfinite(ref_lse)
    assert live.sum() == 5 * 8
    np.testing.assert_allclose(st.m[live] + np.log(st.l[live]), ref_lse[live], atol=1e-12)
    assert np.all(st.l[~live] == 0) and np.all(np.isneginf(st.m[~live]))


def test_full_token_counts_equal_default(oracle_mod):
    case = _small(3)
    a = oracle_mod.DecodeState(case.num_seqs, case.num_q_heads, case.head_dim)
    b = a.copy()
    for t in range(case.num_steps):
        tb, tc = case.tile(t)
        oracle_mod.decode_step(a, case.q, case.k_pool, case.v_pool, tb, tc, case.num_kv_heads,
                               case.block_size)
        oracle_mod.decode_step(b, case.q, case.k_pool, case.v_pool, tb, tc, case.num_kv_heads,
                               case.block_size, tile_token_counts=tc * case.block_size)
    assert np.array_equal(a.m, b.m) and np.array_equal(a.l, b.l) and np.array_equal(a.o, b.o)


def test_token_count_beyond_listed_blocks_rejected(oracle_mod):
    case = _small(4)
    st = oracle_mod.DecodeState(case.num_seqs, case.num_q_heads, case.head_dim)
    tb, tc = case.tile(0)
    with pytest.raises(ValueError):
        oracle_mod.decode_step(st, case.q, case.k_pool, case.v_pool, tb, tc, case.num_kv_heads,
                               case.block_size, tile_token_counts=tc * case.block_size + 1)
