"""Pins for the varlen forward oracle (CPU only).

Each check ties the fp64 oracle to something other than itself:
  * a brute-force numpy formulation (whole masked score matrix, softmax
    without the max shift, lse = log of the plain sum);
  * grouped-query attention (K/V with fewer heads than Q): torch float64
    scaled_dot_product_attention on K/V heads expanded by repeat_interleave;
  * torch float64 scaled_dot_product_attention per sequence (its causal mask
    is tril(ones(L, S)), i.e. top-left) and torch.logsumexp;
  * the worked examples the implementation plan's CPU tests print
    (tests/golden/plan_test*.json);
  * closed forms: one key gives out = v, equal logits give the mean of the
    visible V rows, causal query 0 gives its own v, an empty key set gives
    out = 0 and lse = -FLT_MAX.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from variable_length_flashattention_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FLT_MAX = float(np.finfo(np.float32).max)


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _f64(t):
    return t.to(torch.float64).numpy()


def _brute_force(case):
    """Second formulation: materialise the masked [Lq, Lk] matrix per (sequence, head)."""
    q, k, v = _f64(case.q), _f64(case.k), _f64(case.v)
    H, D = case.num_heads, case.head_dim
    out = np.zeros((case.total_q, H, D))
    lse = np.full((case.total_q, H), -FLT_MAX)
    for b in range(case.batch):
        q0, q1 = case.cu_seqlens_q[b], case.cu_seqlens_q[b + 1]
        k0, k1 = case.cu_seqlens_k[b], case.cu_seqlens_k[b + 1]
        lq, lk = q1 - q0, k1 - k0
        if lq == 0 or lk == 0:
            continue
        for h in range(H):
            s = case.softmax_scale * (q[q0:q1, h, :] @ k[k0:k1, h, :].T)
            assert np.abs(s).max() < 50.0, "brute force form needs small logits"
            e = np.exp(s)
            if case.causal:
                e = e * np.tril(np.ones((lq, lk)))
            z = e.sum(axis=1)
            out[q0:q1, h, :] = (e @ v[k0:k1, h, :]) / z[:, None]
            lse[q0:q1, h] = np.log(z)
    return out, lse


def _case(lq, lk, H, D, causal, seed, sigma=1.0):
    return W.make_varlen("t", lq, lk, H, D, causal, sigma, value_seed=seed)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [
    ([1, 7, 64, 129], [1, 7, 64, 129], 2, 64),     # the tiny workload
    ([5, 1, 33, 17], [9, 3, 33, 2], 3, 16),        # cross lengths, Lq != Lk both ways
    ([0, 4, 3], [2, 0, 6], 2, 8),                  # empty q and empty k sequences
])
def test_matches_brute_force(oracle_mod, causal, shape):
    lq, lk, H, D = shape
    case = _case(lq, lk, H, D, causal, seed=11)
    out, lse, _ = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q,
                                        case.cu_seqlens_k, H, D, case.softmax_scale, causal)
    ref_out, ref_lse = _brute_force(case)
    np.testing.assert_allclose(out, ref_out, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_float64(oracle_mod, causal):
    lq, lk = [3, 40, 17, 1], [3, 25, 60, 1]
    H, D = 4, 32
    case = _case(lq, lk, H, D, causal, seed=5)
    out, lse, _ = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q,
                                        case.cu_seqlens_k, H, D, case.softmax_scale, causal)
    q, k, v = case.q.double(), case.k.double(), case.v.double()
    for b in range(case.batch):
        q0, q1 = int(case.cu_seqlens_q[b]), int(case.cu_seqlens_q[b + 1])
        k0, k1 = int(case.cu_seqlens_k[b]), int(case.cu_seqlens_k[b + 1])
        qs = q[q0:q1].transpose(0, 1)     # [H, Lq, D]
        ks = k[k0:k1].transpose(0, 1)
        vs = v[k0:k1].transpose(0, 1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qs, ks, vs, is_causal=causal, scale=case.softmax_scale)
        np.testing.assert_allclose(out[q0:q1], ref.transpose(0, 1).numpy(), rtol=1e-10, atol=1e-12)
        s = case.softmax_scale * (qs @ ks.transpose(1, 2))
        if causal:
            s = s.masked_fill(~torch.ones(q1 - q0, k1 - k0, dtype=torch.bool).tril(), float("-inf"))
        ref_lse = torch.logsumexp(s, dim=-1).transpose(0, 1).numpy()
        np.testing.assert_allclose(lse[q0:q1], ref_lse, rtol=1e-12, atol=1e-12)


def test_rows_api_matches_full(oracle_mod):
    case = _case([20, 1, 70], [31, 5, 70], 3, 16, True, seed=3)
    out, lse, _ = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q,
                                        case.cu_seqlens_k, 3, 16, case.softmax_scale, True)
    rng = np.random.default_rng(0)
    rows = np.stack([rng.integers(0, case.total_q, 50), rng.integers(0, 3, 50)], axis=1)
    ro, rl, _ = oracle_mod.varlen_fwd_rows(case.q, case.k, case.v, case.cu_seqlens_q,
                                           case.cu_seqlens_k, 3, 16, case.softmax_scale, True, rows)
    np.testing.assert_array_equal(ro, out[rows[:, 0], rows[:, 1]])
    np.testing.assert_array_equal(rl, lse[rows[:, 0], rows[:, 1]])


def _const_case(cu, H, D, token_values):
    """q = k = v = token_values[t] in every (head, dim)."""
    cu = np.asarray(cu, dtype=np.int32)
    x = torch.tensor(token_values, dtype=torch.float32)[:, None, None].expand(-1, H, D)
    x = x.contiguous().to(torch.bfloat16)
    return cu, x


def test_plan_example_two_sequences_independent(oracle_mod):
    g = _golden("plan_test2_two_sequences_independent.json")
    H, D = g["num_heads"], g["head_dim"]
    cu, x = _const_case(g["cu_seqlens"], H, D, g["token_value"])
    out, _, _ = oracle_mod.varlen_fwd(x, x, x, cu, cu, H, D, g["softmax_scale"], g["causal"])
    for t, want in enumerate(g["expected_out_per_token"]):
        assert np.all(np.abs(out[t] - want) < g["abs_tol"])


def test_plan_example_causal_mask(oracle_mod):
    g = _golden("plan_test5_causal_mask.json")
    H, D = g["num_heads"], g["head_dim"]
    cu = np.asarray(g["cu_seqlens"], dtype=np.int32)
    ones = torch.ones(4, H, D, dtype=torch.bfloat16)
    v = torch.tensor(g["v_per_token"])[:, None, None].expand(-1, H, D).contiguous().to(torch.bfloat16)
    oc, _, _ = oracle_mod.varlen_fwd(ones, ones, v, cu, cu, H, D, g["softmax_scale"], True)
    on, _, _ = oracle_mod.varlen_fwd(ones, ones, v, cu, cu, H, D, g["softmax_scale"], False)
    tol = g["abs_tol"]
    assert np.all(np.abs(oc[0] - g["expected_causal_token0"]) < tol)
    assert np.all(np.abs(on[0] - g["expected_noncausal_token0"]) < tol)
    assert np.all(np.abs(oc[-1] - on[-1]) < tol)


def test_plan_example_weights_sum_to_one(oracle_mod):
    g = _golden("plan_test6_weights_sum_to_one.json")
    H, D = g["num_heads"], g["head_dim"]
    cu = np.asarray(g["cu_seqlens"], dtype=np.int32)
    total = int(cu[-1])
    ones = torch.ones(total, H, D, dtype=torch.bfloat16)
    v = torch.zeros(total, H, D)
    for t in range(total):
        v[t, :, t % D] = 1.0
    v = v.to(torch.bfloat16)
    out, _, _ = oracle_mod.varlen_fwd(ones, ones, v, cu, cu, H, D, 1.0 / math.sqrt(D), False)
    for b in range(len(cu) - 1):
        for t in range(cu[b], cu[b + 1]):
            for h in range(H):
                s = sum(out[t, h, kt % D] for kt in range(cu[b], cu[b + 1]))
                assert abs(s - g["expected_weight_sum"]) < g["abs_tol"]


def test_plan_example_empty_sequence(oracle_mod):
    g = _golden("plan_test7_empty_sequence.json")
    H, D = g["num_heads"], g["head_dim"]
    cu = np.asarray(g["cu_seqlens"], dtype=np.int32)
    x = torch.full((int(cu[-1]), H, D), g["value"], dtype=torch.bfloat16)
    out, lse, _ = oracle_mod.varlen_fwd(x, x, x, cu, cu, H, D, g["softmax_scale"], g["causal"])
    assert np.all(np.isfinite(out))
    assert np.all(np.abs(out - g["expected_out"]) < g["abs_tol"])


def test_single_key_gives_v(oracle_mod):
    case = _case([5, 9, 1], [1, 1, 1], 2, 16, False, seed=2)
    out, lse, _ = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q,
                                        case.cu_seqlens_k, 2, 16, case.softmax_scale, False)
    v = _f64(case.v)
    q, k = _f64(case.q), _f64(case.k)
    for b in range(case.batch):
        for t in range(case.cu_seqlens_q[b], case.cu_seqlens_q[b + 1]):
            np.testing.assert_array_equal(out[t], v[b])        # one key: its weight is exactly 1
            s = case.softmax_scale * np.sum(q[t] * k[b], axis=-1)
            np.testing.assert_allclose(lse[t], s, rtol=1e-13, atol=1e-13)   # lse = the one logit


@pytest.mark.parametrize("causal", [False, True])
def test_equal_logits_give_mean_of_visible_v(oracle_mod, causal):
    lq, lk = [6, 13], [6, 13]
    H, D = 2, 8
    case = _case(lq, lk, H, D, causal, seed=4)
    zeros = torch.zeros_like(case.q)              # q = 0: every logit is 0
    out, lse, _ = oracle_mod.varlen_fwd(zeros, case.k, case.v, case.cu_seqlens_q,
                                        case.cu_seqlens_k, H, D, case.softmax_scale, causal)
    v = _f64(case.v)
    for b in range(case.batch):
        k0 = case.cu_seqlens_k[b]
        for i in range(lq[b]):
            t = case.cu_seqlens_q[b] + i
            n = min(i + 1, lk[b]) if causal else lk[b]
            np.testing.assert_allclose(out[t], v[k0:k0 + n].mean(axis=0), rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(lse[t], math.log(n), rtol=1e-14)


def test_causal_query0_gives_its_v0(oracle_mod):
    case = _case([4, 30, 2], [4, 30, 2], 3, 16, True, seed=8)
    out, _, _ = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q,
                                      case.cu_seqlens_k, 3, 16, case.softmax_scale, True)
    v = _f64(case.v)
    for b in range(case.batch):
        np.testing.assert_array_equal(out[case.cu_seqlens_q[b]], v[case.cu_seqlens_k[b]])


def test_empty_key_set_gives_zero_and_flt_max(oracle_mod):
    case = _case([3, 2], [0, 4], 2, 8, False, seed=1)
    out, lse, _ = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q,
                                        case.cu_seqlens_k, 2, 8, case.softmax_scale, False)
    assert np.all(out[:3] == 0.0)
    assert np.all(lse[:3] == -FLT_MAX)
    assert np.all(np.isfinite(lse[3:])) and np.all(lse[3:] > -1e30)


def test_packed_equals_each_sequence_alone(oracle_mod):
    lq, lk = [7, 12, 3], [9, 12, 5]
    case = _case(lq, lk, 2, 16, True, seed=6)
    out, lse, _ = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q,
                                        case.cu_seqlens_k, 2, 16, case.softmax_scale, True)
    for b in range(case.batch):
        q0, q1 = case.cu_seqlens_q[b], case.cu_seqlens_q[b + 1]
        k0, k1 = case.cu_seqlens_k[b], case.cu_seqlens_k[b + 1]
        cq = np.array([0, q1 - q0], dtype=np.int32)
        ck = np.array([0, k1 - k0], dtype=np.int32)
        o1, l1, _ = oracle_mod.varlen_fwd(case.q[q0:q1], case.k[k0:k1], case.v[k0:k1], cq, ck,
                                          2, 16, case.softmax_scale, True)
        np.testing.assert_array_equal(out[q0:q1], o1)
        np.testing.assert_array_equal(lse[q0:q1], l1)


def test_thread_count_does_not_change_result(oracle_mod):
    case = W.tiny(True, seed=1)
    a = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q, case.cu_seqlens_k,
                              2, 64, case.softmax_scale, True, nthreads=1)
    b = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q, case.cu_seqlens_k,
                              2, 64, case.softmax_scale, True, nthreads=4)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_rejects_bad_cu_seqlens(oracle_mod):
    x = torch.ones(4, 1, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        oracle_mod.varlen_fwd(x, x, x, np.array([1, 4], np.int32), np.array([0, 4], np.int32),
                              1, 8, 0.5, False)


@pytest.mark.parametrize("Hkv", [1, 2])
@pytest.mark.parametrize("causal", [False, True])
def test_grouped_kv_heads_match_torch_sdpa_float64(oracle_mod, causal, Hkv):
    lq, lk = [3, 40, 17, 1], [3, 25, 60, 1]
    H, D = 8, 32
    case = _case(lq, lk, H, D, causal, seed=11)
    k = case.k[:, :Hkv].contiguous()           # K/V with Hkv heads
    v = case.v[:, :Hkv].contiguous()
    out, lse, _ = oracle_mod.varlen_fwd(case.q, k, v, case.cu_seqlens_q, case.cu_seqlens_k, H, D,
                                        case.softmax_scale, causal, num_kv_heads=Hkv)
    g = H // Hkv
    q, kd, vd = case.q.double(), k.double(), v.double()
    for b in range(case.batch):
        q0, q1 = int(case.cu_seqlens_q[b]), int(case.cu_seqlens_q[b + 1])
        k0, k1 = int(case.cu_seqlens_k[b]), int(case.cu_seqlens_k[b + 1])
        qs = q[q0:q1].transpose(0, 1)
        ks = kd[k0:k1].repeat_interleave(g, dim=1).transpose(0, 1)   # head h <- kv head h // g
        vs = vd[k0:k1].repeat_interleave(g, dim=1).transpose(0, 1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qs, ks, vs, is_causal=causal, scale=case.softmax_scale)
        np.testing.assert_allclose(out[q0:q1], ref.transpose(0, 1).numpy(), rtol=1e-10, atol=1e-12)
        s_ = case.softmax_scale * (qs @ ks.transpose(1, 2))
        if causal:
            s_ = s_.masked_fill(~torch.ones(q1 - q0, k1 - k0, dtype=torch.bool).tril(),
                                float("-inf"))
        np.testing.assert_allclose(lse[q0:q1], torch.logsumexp(s_, dim=-1).transpose(0, 1).numpy(),
                                   rtol=1e-12, atol=1e-12)
    rng = np.random.default_rng(1)
    rows = np.stack([rng.integers(0, case.total_q, 40), rng.integers(0, H, 40)], axis=1)
    ro, rl, _ = oracle_mod.varlen_fwd_rows(case.q, k, v, case.cu_seqlens_q, case.cu_seqlens_k, H,
                                           D, case.softmax_scale, causal, rows, num_kv_heads=Hkv)
    np.testing.assert_array_equal(ro, out[rows[:, 0], rows[:, 1]])
    np.testing.assert_array_equal(rl, lse[rows[:, 0], rows[:, 1]])


def test_bottom_right_causal_matches_torch_sdpa_float64(oracle_mod):
    # causal == 2: local key j visible to local query i iff j <= i + Lk - Lq
    lq, lk = [3, 40, 60, 1, 25], [3, 25, 17, 9, 0]
    H, D = 4, 32
    case = _case(lq, lk, H, D, True, seed=13)
    out, lse, _ = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q,
                                        case.cu_seqlens_k, H, D, case.softmax_scale, 2)
    q, k, v = case.q.double(), case.k.double(), case.v.double()
    for b in range(case.batch):
        q0, q1 = int(case.cu_seqlens_q[b]), int(case.cu_seqlens_q[b + 1])
        k0, k1 = int(case.cu_seqlens_k[b]), int(case.cu_seqlens_k[b + 1])
        Lq, Lk = q1 - q0, k1 - k0
        allowed = torch.ones(Lq, Lk, dtype=torch.bool).tril(diagonal=Lk - Lq)
        for r in range(Lq):
            if Lk == 0 or not allowed[r].any():
                assert np.all(out[q0 + r] == 0) and np.all(lse[q0 + r] == -oracle_mod.FLT_MAX)
        live = allowed.any(dim=1)
        if not live.any():
            continue
        qs = q[q0:q1].transpose(0, 1)[:, live]
        ks = k[k0:k1].transpose(0, 1)
        vs = v[k0:k1].transpose(0, 1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qs, ks, vs, attn_mask=allowed[live], scale=case.softmax_scale)
        np.testing.assert_allclose(out[q0:q1][live.numpy()], ref.transpose(0, 1).numpy(),
                                   rtol=1e-10, atol=1e-12)
        s_ = (case.softmax_scale * (qs @ ks.transpose(1, 2))).masked_fill(~allowed[live],
                                                                          float("-inf"))
        np.testing.assert_allclose(lse[q0:q1][live.numpy()],
                                   torch.logsumexp(s_, dim=-1).transpose(0, 1).numpy(),
                                   rtol=1e-12, atol=1e-12)


def _band(Lq, Lk, causal, window_left):
    """Visible-key mask of one sequence: j <= i + off, and j >= i + off - window_left."""
    off = Lk - Lq if causal == 2 else 0
    i = torch.arange(Lq)[:, None]
    j = torch.arange(Lk)[None, :]
    allowed = j <= i + off
    if window_left >= 0:
        allowed &= j >= i + off - window_left
    return allowed


@pytest.mark.parametrize("causal", [1, 2])
@pytest.mark.parametrize("window_left", [0, 3, 37, 130])
def test_sliding_window_matches_torch_sdpa_float64(oracle_mod, causal, window_left):
    # keys j with i + off - window_left <= j <= i + off, the rest weight zero
    lq, lk = [3, 140, 60, 1, 25, 200], [3, 170, 17, 9, 0, 90]
    H, D = 2, 32
    case = _case(lq, lk, H, D, True, seed=17 + window_left)
    out, lse, _ = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q,
                                        case.cu_seqlens_k, H, D, case.softmax_scale, causal,
                                        window_left=window_left)
    q, k, v = case.q.double(), case.k.double(), case.v.double()
    for b in range(case.batch):
        q0, q1 = int(case.cu_seqlens_q[b]), int(case.cu_seqlens_q[b + 1])
        k0, k1 = int(case.cu_seqlens_k[b]), int(case.cu_seqlens_k[b + 1])
        allowed = _band(q1 - q0, k1 - k0, causal, window_left)
        live = allowed.any(dim=1) if k1 > k0 else torch.zeros(q1 - q0, dtype=torch.bool)
        dead = ~live.numpy()
        assert np.all(out[q0:q1][dead] == 0) and np.all(lse[q0:q1][dead] == -oracle_mod.FLT_MAX)
        if not live.any():
            continue
        qs = q[q0:q1].transpose(0, 1)[:, live]
        ks = k[k0:k1].transpose(0, 1)
        vs = v[k0:k1].transpose(0, 1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qs, ks, vs, attn_mask=allowed[live], scale=case.softmax_scale)
        np.testing.assert_allclose(out[q0:q1][live.numpy()], ref.transpose(0, 1).numpy(),
                                   rtol=1e-10, atol=1e-12)
        s_ = (case.softmax_scale * (qs @ ks.transpose(1, 2))).masked_fill(~allowed[live],
                                                                          float("-inf"))
        np.testing.assert_allclose(lse[q0:q1][live.numpy()],
                                   torch.logsumexp(s_, dim=-1).transpose(0, 1).numpy(),
                                   rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [1, 2])
def test_zero_window_gives_the_diagonal_v(oracle_mod, causal):
    # window_left = 0: the only visible key is j = i + off, weight exactly 1,
    # so out is that key's v row and lse its scaled score
    lq, lk = [5, 40, 1], [9, 40, 4]
    H, D = 2, 16
    case = _case(lq, lk, H, D, True, seed=23)
    out, lse, _ = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q,
                                        case.cu_seqlens_k, H, D, case.softmax_scale, causal,
                                        window_left=0)
    q, k, v = _f64(case.q), _f64(case.k), _f64(case.v)
    for b in range(case.batch):
        q0, k0 = int(case.cu_seqlens_q[b]), int(case.cu_seqlens_k[b])
        off = lk[b] - lq[b] if causal == 2 else 0
        for i in range(lq[b]):
            j = i + off
            if not 0 <= j < lk[b]:
                assert np.all(out[q0 + i] == 0)
                continue
            np.testing.assert_array_equal(out[q0 + i], v[k0 + j])
            s = case.softmax_scale * np.einsum("hd,hd->h", q[q0 + i], k[k0 + j])
            np.testing.assert_allclose(lse[q0 + i], s, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("causal", [1, 2])
def test_window_wider_than_keys_changes_nothing(oracle_mod, causal):
    lq, lk = [70, 3, 128], [70, 50, 100]
    case = _case(lq, lk, 2, 32, True, seed=29)
    args = (case.q, case.k, case.v, case.cu_seqlens_q, case.cu_seqlens_k, 2, 32,
            case.softmax_scale, causal)
    o0, l0, _ = oracle_mod.varlen_fwd(*args)
    o1, l1, _ = oracle_mod.varlen_fwd(*args, window_left=max(lq) + max(lk))
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(l0, l1)


def test_window_needs_a_causal_mode(oracle_mod):
    case = _case([4], [4], 1, 16, False, seed=1)
    with pytest.raises(ValueError):
        oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q, case.cu_seqlens_k, 1, 16,
                              case.softmax_scale, 0, window_left=2)
