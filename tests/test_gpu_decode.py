"""GPU parity of the paged GQA decode (init, step, finalize) against the fp64
oracle, the block-table gather bit-exact against a CPU gather, and the
device-side checks of block ids and counts."""
import math

import numpy as np
import pytest
import torch

from helpers import assert_out_close
from variable_length_flashattention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vfa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from variable_length_flashattention_gb300 import build, vfa as binding
    build.build()
    return binding


def _gpu_state(case):
    S, Hq, D = case.num_seqs, case.num_q_heads, case.head_dim
    m = torch.empty(S, Hq, device="cuda")
    l = torch.empty(S, Hq, device="cuda")
    o = torch.empty(S, Hq, D, device="cuda")
    return m, l, o


def _run_gpu(vfa, case, status=None, exact=False, scale=0.0):
    m, l, o = _gpu_state(case)
    q, kp, vp = case.q.cuda(), case.k_pool.cuda(), case.v_pool.cuda()
    vfa.decode_init(m, l, o, status)
    for t in range(case.num_steps):
        tb, tc = case.tile(t)
        tt = torch.from_numpy(case.tile_tokens(t)).cuda() if exact else None
        vfa.decode_step(q, kp, vp, torch.from_numpy(tb).cuda(), torch.from_numpy(tc).cuda(),
                        m, l, o, status, tile_token_counts=tt, softmax_scale=scale)
    out = vfa.decode_finalize(l, o)
    torch.cuda.synchronize()
    return m.cpu().double().numpy(), l.cpu().double().numpy(), o.cpu().double().numpy(), \
        out.float().cpu().double().numpy()


def _run_oracle(oracle_mod, case, exact=False, scale=0.0):
    st = oracle_mod.DecodeState(case.num_seqs, case.num_q_heads, case.head_dim)
    for t in range(case.num_steps):
        tb, tc = case.tile(t)
        oracle_mod.decode_step(st, case.q, case.k_pool, case.v_pool, tb, tc, case.num_kv_heads,
                               case.block_size,
                               tile_token_counts=case.tile_tokens(t) if exact else None,
                               scale=scale)
    return st, oracle_mod.decode_finalize(st)


def _compare(m, l, o, out, st, ref, what):
    assert_out_close(out, ref, what + " out")
    live = st.l > 0
    assert np.all(l[~live] == 0) and np.all(np.isneginf(m[~live]))
    lse_gpu = m[live] + np.log(l[live])
    lse_ref = st.m[live] + np.log(st.l[live])
    assert np.abs(lse_gpu - lse_ref).max() <= 2e-3, f"{what}: state m + ln l"
    assert_out_close(o[live] / l[live][:, None], ref[live], what + " o/l")


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_decode_workload(vfa, oracle_mod, seed):
    case = W.decode(seed)
    assert case.num_steps <= 16 and case.num_seqs == 64
    m, l, o, out = _run_gpu(vfa, case)
    st, ref = _run_oracle(oracle_mod, case)
    _compare(m, l, o, out, st, ref, "decode")


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 8, 64), (8, 4, 128), (32, 8, 128), (16, 2, 256),
                                      (4, 1, 64), (8, 1, 256), (8, 1, 128), (8, 1, 64),
                                      (2, 2, 256), (3, 3, 128), (4, 2, 64), (4, 2, 256)])
def test_decode_shapes(vfa, oracle_mod, Hq, Hkv, D):
    rng = np.random.default_rng(Hq * 100 + D)
    n_blocks = [5, 0, 1, 13, 7]
    perm = rng.permutation(sum(n_blocks)).astype(np.int32)
    case = W.make_decode("shapes", n_blocks, Hq, Hkv, D, 16, 3, perm, value_seed=D + Hkv)
    m, l, o, out = _run_gpu(vfa, case)
    st, ref = _run_oracle(oracle_mod, case)
    _compare(m, l, o, out, st, ref, f"decode {Hq}/{Hkv}/{D}")


def test_tile_split_invariance_on_gpu(vfa, oracle_mod):
    rng = np.random.default_rng(7)
    n_blocks = [40, 3, 17]
    perm = rng.permutation(sum(n_blocks)).astype(np.int32)
    outs = []
    for cap in (1, 5, 32, 64):
        case = W.make_decode("split", n_blocks, 8, 2, 128, 16, cap, perm, value_seed=1)
        outs.append(_run_gpu(vfa, case)[3])
    st, ref = _run_oracle(oracle_mod, W.make_decode("split", n_blocks, 8, 2, 128, 16, 64, perm,
                                                    value_seed=1))
    for out in outs:
        assert_out_close(out, ref, "split")


def test_gather_bit_exact(vfa):
    case = W.decode(1, num_seqs=6, ctx_lo=16, ctx_hi=600)
    S, cap, bs, Hkv, D = case.num_seqs, case.tile_capacity, 16, case.num_kv_heads, case.head_dim
    kp, vp = case.k_pool.cuda(), case.v_pool.cuda()
    for t in range(case.num_steps):
        tb, tc = case.tile(t)
        k_out = torch.zeros(S, cap, bs, Hkv, D, dtype=torch.bfloat16, device="cuda")
        v_out = torch.zeros_like(k_out)
        vfa.debug_paged_gather(kp, vp, torch.from_numpy(tb).cuda(), torch.from_numpy(tc).cuda(),
                               k_out, v_out)
        kg = k_out.cpu().view(torch.int16).numpy()
        vg = v_out.cpu().view(torch.int16).numpy()
        kpool = case.k_pool.view(torch.int16).numpy()
        vpool = case.v_pool.view(torch.int16).numpy()
        for s in range(S):
            n = int(tc[s])
            np.testing.assert_array_equal(kg[s, :n], kpool[tb[s, :n]])
            np.testing.assert_array_equal(vg[s, :n], vpool[tb[s, :n]])
            assert np.all(kg[s, n:] == 0) and np.all(vg[s, n:] == 0)


def test_one_hot_v_pins_which_tokens_are_read(vfa):
    # K = 0: every token gets the same weight, so out = mean of the gathered V rows;
    # V row of pool token (blk, t) is one-hot at column (blk * 16 + t) % D.
    n_blocks = [3, 1, 2]
    nb = sum(n_blocks)
    Hq, Hkv, D = 4, 1, 128
    rng = np.random.default_rng(3)
    perm = rng.permutation(nb).astype(np.int32)
    case = W.make_decode("onehot", n_blocks, Hq, Hkv, D, 16, 32, perm, value_seed=0)
    k = torch.zeros_like(case.k_pool)
    v = torch.zeros(nb, 16, Hkv, D)
    for blk in range(nb):
        for t in range(16):
            v[blk, t, 0, (blk * 16 + t) % D] = 1.0
    case = W.DecodeCase(case.name, case.context_lengths, n_blocks, Hq, Hkv, D, 16, 32, case.q,
                        k, v.to(torch.bfloat16), case.block_table)
    _, _, _, out = _run_gpu(vfa, case)
    for s, ids in enumerate(case.block_table):
        want = np.zeros(D)
        for blk in ids:
            for t in range(16):
                want[(blk * 16 + t) % D] += 1.0 / (16 * len(ids))
        for qh in range(Hq):
            np.testing.assert_allclose(out[s, qh], want, atol=2e-3)


@pytest.mark.parametrize("bad", ["block_id", "negative_id", "count"])
def test_bad_block_table_sets_status_and_skips_sequence(vfa, bad):
    n_blocks = [4, 4]
    rng = np.random.default_rng(0)
    case = W.make_decode("bad", n_blocks, 8, 2, 128, 16, 4, rng.permutation(8).astype(np.int32),
                         value_seed=2)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    m, l, o = _gpu_state(case)
    vfa.decode_init(m, l, o, status)
    assert vfa.read_status(status) == 0
    tb, tc = case.tile(0)
    if bad == "block_id":
        tb[1, 2] = case.num_blocks
    elif bad == "negative_id":
        tb[1, 0] = -3
    else:
        tc[1] = 5
    vfa.decode_step(case.q.cuda(), case.k_pool.cuda(), case.v_pool.cuda(),
                    torch.from_numpy(tb).cuda(), torch.from_numpy(tc).cuda(), m, l, o, status)
    assert vfa.read_status(status) == vfa.VFA_ERR_BAD_BLOCK
    assert torch.all(torch.isneginf(m[1])) and torch.all(l[1] == 0) and torch.all(o[1] == 0)
    assert torch.all(l[0] > 0)                     # the valid sequence was still updated


# Contexts that end inside their last block, and an explicit scale: the step
# absorbs only the first tile_token_counts[s] tokens of the listed blocks.

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_decode_workload_exact_context(vfa, oracle_mod, seed):
    case = W.decode(seed)
    assert any(c % case.block_size for c in case.context_lengths)
    m, l, o, out = _run_gpu(vfa, case, exact=True)
    st, ref = _run_oracle(oracle_mod, case, exact=True)
    _compare(m, l, o, out, st, ref, "decode exact context")


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 8, 64), (32, 8, 128), (8, 1, 128), (16, 2, 256),
                                      (4, 2, 64)])
@pytest.mark.parametrize("scale", [0.0, 0.05])
def test_decode_exact_context_shapes(vfa, oracle_mod, Hq, Hkv, D, scale):
    rng = np.random.default_rng(Hq + D)
    n_blocks = [5, 0, 1, 13, 7, 3]
    ctx = [5 * 16 - 3, 0, 1, 13 * 16, 7 * 16 - 15, 33]       # 33: last listed block unread
    perm = rng.permutation(sum(n_blocks)).astype(np.int32)
    case = W.make_decode("exact", n_blocks, Hq, Hkv, D, 16, 3, perm, value_seed=D + Hq,
                         context_lengths=ctx)
    m, l, o, out = _run_gpu(vfa, case, exact=True, scale=scale)
    st, ref = _run_oracle(oracle_mod, case, exact=True, scale=scale)
    _compare(m, l, o, out, st, ref, f"decode exact {Hq}/{Hkv}/{D} scale {scale}")


def test_bad_token_count_sets_status_and_skips_sequence(vfa):
    case = W.make_decode("badtok", [2, 2], 4, 2, 64, 16, 2, np.arange(4, dtype=np.int32), 3)
    m, l, o = _gpu_state(case)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    vfa.decode_init(m, l, o, status)
    tb, tc = case.tile(0)
    tt = torch.tensor([2 * 16 + 1, 20], dtype=torch.int32, device="cuda")   # seq 0: too many
    vfa.decode_step(case.q.cuda(), case.k_pool.cuda(), case.v_pool.cuda(),
                    torch.from_numpy(tb).cuda(), torch.from_numpy(tc).cuda(), m, l, o, status,
                    tile_token_counts=tt)
    torch.cuda.synchronize()
    assert int(status.item()) == vfa.VFA_ERR_BAD_BLOCK
    assert torch.all(torch.isneginf(m[0])) and torch.all(l[0] == 0)      # left as it was
    assert torch.all(torch.isfinite(m[1])) and torch.all(l[1] > 0)       # the valid one ran


# Split step: each (sequence, kv head) tile cut into runs of blocks, one CTA
# each, merged by the last CTA of the row.  The result is the step's state
# update whatever the cut ("attention_ref.rs": tile fragmentation must give
# the single-shot result), checked against the oracle's single-shot state.

def _run_gpu_split(vfa, case, num_splits, exact=False, status=None, ws=None):
    m, l, o = _gpu_state(case)
    q, kp, vp = case.q.cuda(), case.k_pool.cuda(), case.v_pool.cuda()
    S, Hq, Hkv, D = case.num_seqs, case.num_q_heads, case.num_kv_heads, case.head_dim
    if ws is None:
        ws = vfa.alloc_decode_split_workspace(S, Hq, Hkv, D, num_splits)
    vfa.decode_init(m, l, o, status)
    for t in range(case.num_steps):
        tb, tc = case.tile(t)
        tt = torch.from_numpy(case.tile_tokens(t)).cuda() if exact else None
        vfa.decode_step_split(q, kp, vp, torch.from_numpy(tb).cuda(),
                              torch.from_numpy(tc).cuda(), m, l, o, num_splits, ws, status,
                              tile_token_counts=tt)
    out = vfa.decode_finalize(l, o)
    torch.cuda.synchronize()
    return (m.cpu().double().numpy(), l.cpu().double().numpy(), o.cpu().double().numpy(),
            out.float().cpu().double().numpy(), ws)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_split_decode_long_contexts(vfa, oracle_mod, seed):
    # four contexts of 49k-64k tokens, each in one tile of up to 4096 blocks:
    # without the split the step has only 32 CTAs for 152 SMs
    case = W.decode_long(seed)
    assert case.num_steps == 1 and max(case.context_lengths) == 65536
    n = vfa.decode_split_count(case.num_seqs, case.num_kv_heads, case.tile_capacity)
    assert n > 1
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    m, l, o, out, ws = _run_gpu_split(vfa, case, n, exact=True, status=status)
    assert int(status.item()) == 0
    st, ref = _run_oracle(oracle_mod, case, exact=True)
    _compare(m, l, o, out, st, ref, f"split decode long x{n}")
    tickets = ws[:4 * case.num_seqs * case.num_kv_heads].view(torch.int32)
    assert torch.all(tickets == 0)                   # left ready for the next call


@pytest.mark.parametrize("num_splits", [2, 7, 40])
def test_split_decode_workload_steps(vfa, oracle_mod, num_splits):
    # the 64-sequence workload, every 32-block step split (40 runs: most of them
    # empty), chained on one workspace through all steps
    case = W.decode(0)
    m, l, o, out, _ = _run_gpu_split(vfa, case, num_splits)
    st, ref = _run_oracle(oracle_mod, case)
    _compare(m, l, o, out, st, ref, f"split decode x{num_splits}")


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 8, 64), (8, 1, 128), (16, 2, 256), (4, 2, 64)])
def test_split_decode_shapes_exact_context(vfa, oracle_mod, Hq, Hkv, D):
    rng = np.random.default_rng(Hq + D + 1)
    n_blocks = [50, 0, 1, 130, 7, 3]
    ctx = [50 * 16 - 3, 0, 1, 130 * 16, 7 * 16 - 15, 33]
    perm = rng.permutation(sum(n_blocks)).astype(np.int32)
    case = W.make_decode("split-exact", n_blocks, Hq, Hkv, D, 16, 64, perm, value_seed=D + Hq,
                         context_lengths=ctx)
    m, l, o, out, _ = _run_gpu_split(vfa, case, 5, exact=True)
    st, ref = _run_oracle(oracle_mod, case, exact=True)
    _compare(m, l, o, out, st, ref, f"split exact {Hq}/{Hkv}/{D}")


def test_split_decode_bad_block_skips_row_and_keeps_tickets(vfa):
    n_blocks = [20, 20]
    rng = np.random.default_rng(4)
    case = W.make_decode("bad-split", n_blocks, 8, 2, 128, 16, 20,
                         rng.permutation(40).astype(np.int32), value_seed=3)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    m, l, o = _gpu_state(case)
    ws = vfa.alloc_decode_split_workspace(2, 8, 2, 128, 4)
    vfa.decode_init(m, l, o, status)
    tb, tc = case.tile(0)
    tb[1, 13] = case.num_blocks                      # out of the pool
    vfa.decode_step_split(case.q.cuda(), case.k_pool.cuda(), case.v_pool.cuda(),
                          torch.from_numpy(tb).cuda(), torch.from_numpy(tc).cuda(), m, l, o, 4,
                          ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == vfa.VFA_ERR_BAD_BLOCK
    assert torch.all(torch.isneginf(m[1])) and torch.all(l[1] == 0) and torch.all(o[1] == 0)
    assert torch.all(l[0] > 0)
    assert torch.all(ws[:16].view(torch.int32) == 0)
