"""Per-element error bound for the backward's gradients (test-side error model).

The backward rounds four kinds of quantity to bf16 (8 significand bits, so
unit roundoff u = 2^-8 with round to nearest even):
  * P, for the dV = P^T dO product;
  * dS = P (dP - Delta), for the dK = dS^T Q and dQ = dS K products;
  * the forward's out, from which Delta = sum_d dO * out is taken (out
    carries its own rounding and that of the forward's bf16 P);
  * the gradients themselves.
Everything else (the tensor core's fp32 sums of exact bf16 products, ex2 on
fp32 scores, the fp32 lse) contributes relative errors of order 1e-5, far
below u.  To first order each gradient element's error is then
    (final rounding, at most u |exact|)  +  sum_t c_t e_t,
a linear combination of the individual rounding errors e_t (|e_t| <= u) of
P, dS and out, with coefficients c_t given by the exact quantities:
  dV[j]:  c = P_ij dO_i                                 (over queries i)
  Delta_i:  c = dO_id O_id (over d, out rounding) and P_ij dP_ij (over j,
            the forward's P rounding), so dDelta_i is itself such a sum;
  dK[j]:  c = scale q_i dS_ij, and scale q_i P_ij times Delta_i's c's;
  dQ[i]:  c = scale k_j dS_ij, and scale k_j P_ij times Delta_i's c's.
Two bounds on |sum_t c_t e_t| follow:
  * worst case: u M with M = sum_t |c_t| (every error at its extreme, same sign);
  * probabilistic (Higham and Mary, "A new approach to probabilistic rounding
    error analysis", SIAM J. Sci. Comput. 41(5), 2019: rounding errors taken
    as independent, mean zero, bounded by u): by Hoeffding's inequality
    |sum_t c_t e_t| <= lam u R, R = sqrt(sum_t c_t^2), except with probability
    at most 2 exp(-lam^2 / 2); lam = 7 makes that 5e-11 per element.
The tests hold every element to
    |got - ref| <= BWD_FACTOR * u * (|ref| + min(M, lam R)) + BWD_FLOOR,
BWD_FACTOR = 1.5 leaving room for the first-order terms left out.  A float32
emulation of the kernel's arithmetic stays within 0.8 of the unscaled bound
(tests/test_bwd_error_model.py).

The sums are computed here in float64 with torch on the CPU from the inputs
and the mask definitions (visible iff j <= i + off for a causal mode, off = 0
top-left or Lk - Lq bottom-right, and j >= i + off - window_left with a
window); this module is a tolerance, not an oracle.
"""
from __future__ import annotations

import numpy as np
import torch

BF16_U = 2.0 ** -8
LAMBDA = 7.0
BWD_FACTOR = 1.5
BWD_FLOOR = 1e-6


def _visible(lq, lk, causal, window_left):
    i = torch.arange(lq, dtype=torch.int64)[:, None]
    j = torch.arange(lk, dtype=torch.int64)[None, :]
    vis = torch.ones(lq, lk, dtype=torch.bool)
    if causal:
        off = 0 if causal == 1 else lk - lq
        vis &= j <= i + off
        if window_left >= 0:
            vis &= j >= i + off - window_left
    return vis


def magnitudes(case, dout, causal, window_left=-1, num_kv_heads=None):
    """Per-element allowance min(M, LAMBDA R) for (dq [Tq,H,D], dk, dv [Tk,Hkv,D]),
    float64 numpy arrays."""
    H, D = case.num_heads, case.head_dim
    hkv = num_kv_heads or case.k.shape[1]
    g = H // hkv
    scale = float(case.softmax_scale)
    q, k, v, do = (t.double() for t in (case.q, case.k, case.v, dout))
    z = lambda shape: torch.zeros(shape, dtype=torch.float64)
    m_dq, m_dk, m_dv = z(q.shape), z(k.shape), z(k.shape)       # worst-case sums
    r_dq, r_dk, r_dv = z(q.shape), z(k.shape), z(k.shape)       # sums of squares
    cq, ck = case.cu_seqlens_q, case.cu_seqlens_k
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
        lq, lk = q1 - q0, k1 - k0
        if lq == 0 or lk == 0:
            continue
        vis = _visible(lq, lk, causal, window_left)
        for kh in range(hkv):
            heads = list(range(kh * g, kh * g + g))
            qb = q[q0:q1, heads].permute(1, 0, 2)            # [g, lq, D]
            dob = do[q0:q1, heads].permute(1, 0, 2)
            kb = k[k0:k1, kh]                                  # [lk, D]
            vb = v[k0:k1, kh]
            s = scale * qb @ kb.T                              # [g, lq, lk]
            s = s.masked_fill(~vis, float("-inf"))
            mx = s.amax(-1, keepdim=True)
            live = torch.isfinite(mx)
            p = torch.where(live, torch.exp(s - torch.where(live, mx, 0.0)), 0.0)
            p = p / p.sum(-1, keepdim=True).clamp_min(1e-300)
            dp = dob @ vb.T
            delta = (p * dp).sum(-1, keepdim=True)
            ds = p * (dp - delta)
            o = p @ vb
            # Delta_i's coefficients: dO_id O_id over d, P_ij dP_ij over j
            e1 = (dob * o).abs().sum(-1, keepdim=True) + (p * dp).abs().sum(-1, keepdim=True)
            e2 = (dob * o).pow(2).sum(-1, keepdim=True) + (p * dp).pow(2).sum(-1, keepdim=True)
            a1 = ds.abs() + p * e1                            # [g, lq, lk]
            a2 = ds.pow(2) + p.pow(2) * e2
            m_dv[k0:k1, kh] += (p.transpose(1, 2) @ dob.abs()).sum(0)
            r_dv[k0:k1, kh] += (p.pow(2).transpose(1, 2) @ dob.pow(2)).sum(0)
            m_dk[k0:k1, kh] += scale * (a1.transpose(1, 2) @ qb.abs()).sum(0)
            r_dk[k0:k1, kh] += scale ** 2 * (a2.transpose(1, 2) @ qb.pow(2)).sum(0)
            m_dq[q0:q1, heads] = (scale * a1 @ kb.abs()).permute(1, 0, 2)
            r_dq[q0:q1, heads] = (scale ** 2 * a2 @ kb.pow(2)).permute(1, 0, 2)
    allow = lambda m, r: torch.minimum(m, LAMBDA * r.sqrt()).numpy()
    return allow(m_dq, r_dq), allow(m_dk, r_dk), allow(m_dv, r_dv)


def check_grad(got, ref, mag, what):
    """|got - ref| <= BWD_FACTOR * u * (|ref| + mag) + BWD_FLOOR elementwise.

    Returns the largest ratio |got - ref| / (u (|ref| + mag) + floor / factor)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite (unwritten?) gradients"
    unit = BF16_U * (np.abs(ref) + mag) + BWD_FLOOR / BWD_FACTOR
    ratio = np.abs(got - ref) / unit
    worst = float(ratio.max()) if ratio.size else 0.0
    bad = ratio > BWD_FACTOR
    if bad.any():
        idx = np.argwhere(bad)[:5].tolist()
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} beyond {BWD_FACTOR} x the "
                             f"rounding bound; worst ratio {worst:.3g}; first {idx}")
    return worst
