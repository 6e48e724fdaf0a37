"""Pins for the varlen backward oracle (CPU only).

The backward is the derivative of the forward's definition; it is tied to
things other than itself:
  * torch float64 autograd through scaled_dot_product_attention (math path:
    matmul, masked softmax, matmul, each differentiated by torch), per
    sequence, with the causal / bottom-right / sliding-window mask as a
    boolean attn_mask and grouped K/V heads expanded by repeat_interleave
    (autograd sums the group's gradients back);
  * invariants of the softmax Jacobian: the rows of dS sum to zero, so the
    keys' dk sum to zero per (sequence, kv head); P's rows sum to one, so
    the keys' dv sum to the sum of dout over the rows that see a key;
  * closed forms: a single visible key gives dq = dk = 0 and dv = dout;
  * central finite differences of a separate numpy fp64 forward (the loss
    sum(out * dout)) at sampled elements of q, k and v.
"""
import numpy as np
import pytest
import torch

from variable_length_flashattention_gb300 import workloads as W


def _case(lq, lk, H, D, seed, Hkv=None):
    case = W.make_varlen("t", lq, lk, H, D, True, 1.0, value_seed=seed)
    if Hkv is not None:
        case.k = case.k[:, :Hkv].contiguous()
        case.v = case.v[:, :Hkv].contiguous()
    g = torch.Generator().manual_seed(seed + 1000)
    dout = torch.randn(case.q.shape, generator=g).to(torch.bfloat16)
    return case, dout


def _mask(Lq, Lk, causal, window_left):
    off = Lk - Lq if causal == 2 else 0
    i = torch.arange(Lq)[:, None]
    j = torch.arange(Lk)[None, :]
    allowed = torch.ones(Lq, Lk, dtype=torch.bool)
    if causal:
        allowed &= j <= i + off
    if window_left >= 0:
        allowed &= j >= i + off - window_left
    return allowed


def _torch_grads(case, dout, causal, window_left, Hkv):
    H = case.num_heads
    g = H // Hkv
    dq = torch.zeros(case.q.shape, dtype=torch.float64)
    dk = torch.zeros(case.k.shape, dtype=torch.float64)
    dv = torch.zeros(case.v.shape, dtype=torch.float64)
    for b in range(case.batch):
        q0, q1 = int(case.cu_seqlens_q[b]), int(case.cu_seqlens_q[b + 1])
        k0, k1 = int(case.cu_seqlens_k[b]), int(case.cu_seqlens_k[b + 1])
        if q1 == q0 or k1 == k0:
            continue
        allowed = _mask(q1 - q0, k1 - k0, causal, window_left)
        live = allowed.any(dim=1)
        if not live.any():
            continue
        q = case.q[q0:q1].double().transpose(0, 1).requires_grad_(True)
        k = case.k[k0:k1].double().transpose(0, 1).requires_grad_(True)
        v = case.v[k0:k1].double().transpose(0, 1).requires_grad_(True)
        ke = k.repeat_interleave(g, dim=0)
        ve = v.repeat_interleave(g, dim=0)
        out = torch.nn.functional.scaled_dot_product_attention(
            q[:, live], ke, ve, attn_mask=allowed[live], scale=case.softmax_scale)
        do = dout[q0:q1].double().transpose(0, 1)[:, live]
        (out * do).sum().backward()
        dq[q0:q1] = q.grad.transpose(0, 1)
        dk[k0:k1] = k.grad.transpose(0, 1)
        dv[k0:k1] = v.grad.transpose(0, 1)
    return dq.numpy(), dk.numpy(), dv.numpy()


@pytest.mark.parametrize("causal,window_left", [(0, -1), (1, -1), (2, -1), (1, 5), (2, 20)])
@pytest.mark.parametrize("Hkv", [3, 1])
def test_matches_torch_autograd_float64(oracle_mod, causal, window_left, Hkv):
    lq, lk = [5, 40, 1, 0, 33, 70], [9, 40, 4, 6, 20, 0]
    case, dout = _case(lq, lk, 3, 16, seed=31 + causal, Hkv=Hkv)
    dq, dk, dv, _ = oracle_mod.varlen_bwd(case.q, case.k, case.v, dout, case.cu_seqlens_q,
                                          case.cu_seqlens_k, 3, 16, case.softmax_scale, causal,
                                          num_kv_heads=Hkv, window_left=window_left)
    rq, rk, rv = _torch_grads(case, dout, causal, window_left, Hkv)
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        np.testing.assert_allclose(got, ref, rtol=1e-9, atol=1e-11)


def test_key_sums(oracle_mod):
    lq, lk = [50, 17, 64], [50, 40, 3]
    H, D = 2, 8
    case, dout = _case(lq, lk, H, D, seed=41)
    for causal in (0, 1, 2):
        dq, dk, dv, _ = oracle_mod.varlen_bwd(case.q, case.k, case.v, dout, case.cu_seqlens_q,
                                              case.cu_seqlens_k, H, D, case.softmax_scale,
                                              causal)
        for b in range(case.batch):
            q0, q1 = int(case.cu_seqlens_q[b]), int(case.cu_seqlens_q[b + 1])
            k0, k1 = int(case.cu_seqlens_k[b]), int(case.cu_seqlens_k[b + 1])
            live = _mask(q1 - q0, k1 - k0, causal, -1).any(dim=1).numpy()
            np.testing.assert_allclose(dk[k0:k1].sum(axis=0), 0.0, atol=1e-10)
            want = dout[q0:q1].double().numpy()[live].sum(axis=0)
            np.testing.assert_allclose(dv[k0:k1].sum(axis=0), want, rtol=1e-12, atol=1e-11)
            # rows that see no key get no gradient
            assert np.all(dq[q0:q1][~live] == 0)


def test_single_key_closed_form(oracle_mod):
    lq, lk = [6], [1]
    case, dout = _case(lq, lk, 2, 16, seed=43)
    dq, dk, dv, _ = oracle_mod.varlen_bwd(case.q, case.k, case.v, dout, case.cu_seqlens_q,
                                          case.cu_seqlens_k, 2, 16, case.softmax_scale, 0)
    assert np.all(np.abs(dq) < 1e-14) and np.all(np.abs(dk) < 1e-14)
    np.testing.assert_allclose(dv[0], dout.double().numpy().sum(axis=0), rtol=1e-14)


def test_rejects_window_without_causal(oracle_mod):
    case, dout = _case([4], [4], 1, 8, seed=1)
    with pytest.raises(ValueError):
        oracle_mod.varlen_bwd(case.q, case.k, case.v, dout, case.cu_seqlens_q, case.cu_seqlens_k,
                              1, 8, case.softmax_scale, 0, window_left=3)


def _np_loss(q, k, v, dout, cu_q, cu_k, scale, causal):
    """L = sum(out * dout) of a plain numpy fp64 forward (whole masked score matrix)."""
    total = 0.0
    for b in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        lq, lk = q1 - q0, k1 - k0
        if lq == 0 or lk == 0:
            continue
        off = lk - lq if causal == 2 else 0
        for h in range(q.shape[1]):
            s = scale * q[q0:q1, h] @ k[k0:k1, h].T
            mask = np.ones((lq, lk), dtype=bool)
            if causal:
                mask = np.arange(lk)[None, :] <= np.arange(lq)[:, None] + off
            s = np.where(mask, s, -np.inf)
            live = mask.any(axis=1)
            e = np.exp(s[live] - s[live].max(axis=1, keepdims=True))
            p = e / e.sum(axis=1, keepdims=True)
            total += float((p @ v[k0:k1, h] * dout[q0:q1, h][live]).sum())
    return total


@pytest.mark.parametrize("causal", [0, 1, 2])
def test_finite_differences(oracle_mod, causal):
    # central differences of a separate numpy fp64 forward against the oracle's gradients
    lq, lk = [3, 5], [4, 5]
    case, dout = _case(lq, lk, 1, 4, seed=61 + causal)
    dq, dk, dv, _ = oracle_mod.varlen_bwd(case.q, case.k, case.v, dout, case.cu_seqlens_q,
                                          case.cu_seqlens_k, 1, 4, case.softmax_scale, causal)
    base = [t.double().numpy().copy() for t in (case.q, case.k, case.v)]
    g = dout.double().numpy()
    cq, ck = [int(x) for x in case.cu_seqlens_q], [int(x) for x in case.cu_seqlens_k]
    eps = 1e-6
    rng = np.random.default_rng(causal)
    for which, grad in enumerate((dq, dk, dv)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, n)) for n in base[which].shape)
            plus = [x.copy() for x in base]
            minus = [x.copy() for x in base]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            fd = (_np_loss(*plus, g, cq, ck, case.softmax_scale, causal) -
                  _np_loss(*minus, g, cq, ck, case.softmax_scale, causal)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (which, idx, fd, grad[idx])
