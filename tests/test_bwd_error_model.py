"""The backward's error model (tests/bwd_error_model.py) checked on the CPU.

A float32 emulation of the GPU backward's arithmetic -- fp32 sums of exact
bf16 products, P and dS rounded to bf16 for the products, Delta taken from
the forward's bf16 out (itself computed with a bf16 P), gradients rounded to
bf16 -- must stay inside the bound the GPU tests apply, against the fp64
oracle's exact gradients.  Planted mistakes of the size a real bug would
make (a 2^-5 relative error in one gradient, a sign error in one row of
dQ, a key row's dV written from its neighbour) must fall outside it.
"""
import numpy as np
import pytest
import torch

from bwd_error_model import _visible, check_grad, magnitudes
from variable_length_flashattention_gb300 import workloads as W


def _bf16(x):
    return x.to(torch.bfloat16).to(torch.float32)


def emulate(case, dout, causal, window_left=-1, hkv=None):
    H, D = case.num_heads, case.head_dim
    hkv = hkv or case.k.shape[1]
    g = H // hkv
    sc = float(case.softmax_scale)
    q, k, v, do = (t.float() for t in (case.q, case.k, case.v, dout))
    dq = torch.zeros_like(q)
    dk = torch.zeros_like(k)
    dv = torch.zeros_like(k)
    cq, ck = case.cu_seqlens_q, case.cu_seqlens_k
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
        if q1 == q0 or k1 == k0:
            continue
        vis = _visible(q1 - q0, k1 - k0, causal, window_left)
        for h in range(H):
            kh = h // g
            s = (q[q0:q1, h] @ k[k0:k1, kh].T) * sc
            s = s.masked_fill(~vis, float("-inf"))
            m = s.amax(-1, keepdim=True)
            live = torch.isfinite(m)
            pu = torch.where(live, torch.exp(s - torch.where(live, m, 0.0)), 0.0)
            l = pu.sum(-1, keepdim=True)
            # forward: O = bf16(P) V / l, rounded to bf16; lse in fp32
            o = _bf16((_bf16(pu) @ v[k0:k1, kh]) / l.clamp_min(1e-30))
            lse = torch.where(live, m + torch.log(l.clamp_min(1e-30)), 0.0)
            p = torch.where(live, torch.exp(s - lse), 0.0)
            dp = do[q0:q1, h] @ v[k0:k1, kh].T
            delta = (do[q0:q1, h] * o).sum(-1, keepdim=True)
            ds = _bf16(p * (dp - delta))
            dv[k0:k1, kh] += _bf16(p).T @ do[q0:q1, h]
            dk[k0:k1, kh] += ds.T @ q[q0:q1, h]
            dq[q0:q1, h] = sc * (ds @ k[k0:k1, kh])
    f = lambda t: _bf16(t).double().numpy()
    return f(dq), f(sc * dk), f(dv)


CASES = [
    ("tiny", lambda: W.tiny(True, 0), 1, -1, None),
    ("tiny-noncausal", lambda: W.tiny(False, 1), 0, -1, None),
    ("mix-bottom-right", lambda: W.make_varlen("mix", [300, 7, 0, 129], [90, 7, 5, 300], 2, 64,
                                               True, 1.0, value_seed=5), 2, -1, None),
    ("window", lambda: W.make_varlen("win", [400, 64], [400, 300], 2, 64, True, 1.0,
                                     value_seed=6), 1, 37, None),
    ("window0", lambda: W.make_varlen("win0", [200], [200], 1, 64, True, 1.0, value_seed=8),
     1, 0, None),
]


def _gqa():
    c = W.make_varlen("gqa", [300, 40], [300, 129], 4, 64, True, 1.0, value_seed=7)
    c.k = c.k[:, :1].contiguous()
    c.v = c.v[:, :1].contiguous()
    return c


CASES.append(("gqa", _gqa, 1, -1, 1))


@pytest.mark.parametrize("name,make,causal,wl,hkv", CASES, ids=[c[0] for c in CASES])
def test_emulated_roundings_stay_inside_the_bound(oracle_mod, name, make, causal, wl, hkv):
    case = make()
    dout = W.upstream_grad(case, 0)
    H = case.num_heads
    got = emulate(case, dout, causal, wl, hkv)
    ref = oracle_mod.varlen_bwd(case.q, case.k, case.v, dout, case.cu_seqlens_q,
                                case.cu_seqlens_k, H, case.head_dim, case.softmax_scale, causal,
                                num_kv_heads=hkv or H, window_left=wl)[:3]
    mags = magnitudes(case, dout, causal, wl, hkv or H)
    worst = [check_grad(g, r, m, f"{nm} {name}")
             for g, r, m, nm in zip(got, ref, mags, ("dq", "dk", "dv"))]
    # the model should be close to tight: the emulation stays within the
    # unscaled bound and reaches a fair part of it (a window of 0 keys is
    # exact: P = 1 on the diagonal, dS = 0)
    assert max(worst) <= 1.0
    if wl != 0:
        assert max(worst) >= 0.3


def test_planted_mistakes_fall_outside_the_bound(oracle_mod):
    case = W.make_varlen("mut", [300, 129, 64], [300, 129, 64], 2, 64, True, 1.0, value_seed=3)
    dout = W.upstream_grad(case, 0)
    dq, dk, dv = emulate(case, dout, 1)
    ref = oracle_mod.varlen_bwd(case.q, case.k, case.v, dout, case.cu_seqlens_q,
                                case.cu_seqlens_k, 2, 64, case.softmax_scale, 1)[:3]
    mq, mk, mv = magnitudes(case, dout, 1)
    check_grad(dq, ref[0], mq, "dq")
    check_grad(dk, ref[1], mk, "dk")
    check_grad(dv, ref[2], mv, "dv")
    # a 2^-5 relative error in each gradient
    for got, r, m, nm in ((dq, ref[0], mq, "dq"), (dk, ref[1], mk, "dk"), (dv, ref[2], mv, "dv")):
        with pytest.raises(AssertionError):
            check_grad(got * (1 + 2.0 ** -5), r, m, nm + " scaled")
    # dq of one query row taken with the wrong sign of its dS
    bad = dq.copy()
    bad[100] = -bad[100]
    with pytest.raises(AssertionError):
        check_grad(bad, ref[0], mq, "dq sign")
    # dv of key row j written from key row j + 1 (an index off by one)
    bad = dv.copy()
    bad[10, 1] = dv[11, 1]
    with pytest.raises(AssertionError):
        check_grad(bad, ref[2], mv, "dv shifted row")
