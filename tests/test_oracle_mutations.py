"""Mutation checks of the oracle's pins (CPU only).

Each case plants one plausible mistake in a copy of the oracle's C source
(a wrong mask bound, a dropped term, a wrong index or sign), builds the
copy, and runs a set of independent checks against it in a subprocess:
torch float64 SDPA (masks, grouped heads), torch float64 autograd (the
backward), torch's float8_e4m3fn decoding, and the decode state's
tile-fragmentation invariance.  The unmutated copy must pass every check
and each mutation must fail at least one, so a mistake of that kind cannot
hide behind the pins.
"""
import json
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHECKS = r'''
import json, sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1])          # the (mutated) oracle copy first
sys.path.insert(1, sys.argv[2])          # the repository, for the input generators
import oracle
assert oracle.__file__.startswith(sys.argv[1])
from variable_length_flashattention_gb300 import workloads as W

def mask(lq, lk, causal, wl):
    off = lk - lq if causal == 2 else 0
    i = torch.arange(lq)[:, None]; j = torch.arange(lk)[None, :]
    m = torch.ones(lq, lk, dtype=torch.bool)
    if causal: m &= j <= i + off
    if wl >= 0: m &= j >= i + off - wl
    return m

def sdpa_err(case, out, q, k, v, causal, wl, g):
    err = 0.0
    for b in range(case.batch):
        q0, q1 = int(case.cu_seqlens_q[b]), int(case.cu_seqlens_q[b + 1])
        k0, k1 = int(case.cu_seqlens_k[b]), int(case.cu_seqlens_k[b + 1])
        if q1 == q0 or k1 == k0: continue
        m = mask(q1 - q0, k1 - k0, causal, wl); live = m.any(1)
        if not live.any(): continue
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[q0:q1].transpose(0, 1)[:, live], k[k0:k1].transpose(0, 1).repeat_interleave(g, 0),
            v[k0:k1].transpose(0, 1).repeat_interleave(g, 0), attn_mask=m[live],
            scale=case.softmax_scale)
        err = max(err, float(np.abs(out[q0:q1][live.numpy()] - ref.transpose(0, 1).numpy()).max()))
    return err

res = {}
lq, lk = [5, 40, 1, 30], [9, 40, 4, 20]
for causal, wl in ((0, -1), (1, -1), (2, -1), (1, 4)):
    case = W.make_varlen("m", lq, lk, 4, 16, bool(causal), 1.0, value_seed=7)
    case.k = case.k[:, :2].contiguous(); case.v = case.v[:, :2].contiguous()
    out, lse, _ = oracle.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q, case.cu_seqlens_k,
                                    4, 16, case.softmax_scale, causal, num_kv_heads=2,
                                    window_left=wl)
    res[f"fwd_{causal}_{wl}"] = sdpa_err(case, out, case.q.double(), case.k.double(),
                                         case.v.double(), causal, wl, 2)
    # lse against torch.logsumexp
    e = 0.0
    for b in range(case.batch):
        q0, q1 = int(case.cu_seqlens_q[b]), int(case.cu_seqlens_q[b + 1])
        k0, k1 = int(case.cu_seqlens_k[b]), int(case.cu_seqlens_k[b + 1])
        m = mask(q1 - q0, k1 - k0, causal, wl); live = m.any(1)
        if q1 == q0 or k1 == k0 or not live.any(): continue
        s = case.softmax_scale * (case.q[q0:q1].double().transpose(0, 1) @
                                  case.k[k0:k1].double().transpose(0, 1).repeat_interleave(2, 0).transpose(1, 2))
        s = s.masked_fill(~m, float("-inf"))[:, live]
        e = max(e, float(np.abs(lse[q0:q1][live.numpy()] - torch.logsumexp(s, -1).transpose(0, 1).numpy()).max()))
    res[f"lse_{causal}_{wl}"] = e

# backward against torch autograd
case = W.make_varlen("mb", [6, 20], [6, 25], 2, 8, True, 1.0, value_seed=3)
dout = W.upstream_grad(case, 3)
for causal in (1, 2):
    dq, dk, dv, _ = oracle.varlen_bwd(case.q, case.k, case.v, dout, case.cu_seqlens_q,
                                      case.cu_seqlens_k, 2, 8, case.softmax_scale, causal)
    err = 0.0
    for b in range(case.batch):
        q0, q1 = int(case.cu_seqlens_q[b]), int(case.cu_seqlens_q[b + 1])
        k0, k1 = int(case.cu_seqlens_k[b]), int(case.cu_seqlens_k[b + 1])
        m = mask(q1 - q0, k1 - k0, causal, -1); live = m.any(1)
        q = case.q[q0:q1].double().transpose(0, 1).requires_grad_(True)
        k = case.k[k0:k1].double().transpose(0, 1).requires_grad_(True)
        v = case.v[k0:k1].double().transpose(0, 1).requires_grad_(True)
        o = torch.nn.functional.scaled_dot_product_attention(q[:, live], k, v, attn_mask=m[live],
                                                             scale=case.softmax_scale)
        (o * dout[q0:q1].double().transpose(0, 1)[:, live]).sum().backward()
        for got, ref in ((dq[q0:q1], q.grad), (dk[k0:k1], k.grad), (dv[k0:k1], v.grad)):
            err = max(err, float(np.abs(got - ref.transpose(0, 1).numpy()).max()))
    res[f"bwd_{causal}"] = err

# FP8 decoder against torch
codes = np.arange(256, dtype=np.uint8)
ours = oracle.fp8_e4m3_decode(codes)
ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
ok = ~np.isnan(ref)
res["fp8"] = float(np.abs(ours[ok] - ref[ok]).max()) + float((np.isnan(ours) != np.isnan(ref)).sum())

# decode: one tile of all blocks vs one block per step
perm = np.random.default_rng(0).permutation(12).astype(np.int32)
outs = []
for cap in (12, 1):
    dc = W.make_decode("md", [5, 7], 4, 2, 16, 4, cap, perm, value_seed=5)
    st = oracle.DecodeState(dc.num_seqs, dc.num_q_heads, dc.head_dim)
    for t in range(dc.num_steps):
        tb, tc = dc.tile(t)
        oracle.decode_step(st, dc.q, dc.k_pool, dc.v_pool, tb, tc, dc.num_kv_heads, dc.block_size)
    outs.append(oracle.decode_finalize(st))
res["decode_tiles"] = float(np.abs(outs[0] - outs[1]).max())
print(json.dumps(res))
'''

TOL = 1e-9

MUTATIONS = [
    ("causal_off_by_one", "if (p->causal && j > i + off)\n            continue;                       /* masked",
     "if (p->causal && j >= i + off)\n            continue;                       /* masked"),
    ("window_edge", "if (p->window_left >= 0 && j < i + off - p->window_left)\n            continue;                       /* left",
     "if (p->window_left >= 0 && j <= i + off - p->window_left)\n            continue;                       /* left"),
    ("lse_without_max", "*lse_out = M + log(Z);", "*lse_out = log(Z);"),
    ("no_normalisation", "out_row[d] = acc / Z;", "out_row[d] = acc;"),
    ("gqa_mapping", "const int kh = h / (H / Hkv);\n    const int64_t tq", "const int kh = h % Hkv;\n    const int64_t tq"),
    ("bottom_right_offset", "const int off = p->causal == 2 ? Lk - Lq : 0;\n\n    int n = 0;",
     "const int off = p->causal == 2 ? Lq - Lk : 0;\n\n    int n = 0;"),
    ("bwd_delta_sign", "const double ds = w[a] * (dp[a] - delta);", "const double ds = w[a] * (dp[a] + delta);"),
    ("bwd_dk_scale", "dk_row[d] += p->scale * ds *", "dk_row[d] += ds *"),
    ("bwd_dv_weight", "dv_row[d] += w[a] * bf16_to_double", "dv_row[d] += bf16_to_double"),
    ("fp8_bias", "mag = ldexp(1.0 + (double)m / 8.0, e - 7);", "mag = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("decode_no_carry", "const double carry = exp(m_old - m_new);", "const double carry = 1.0;"),
]


def _copy_oracle(dst, mutation=None):
    os.makedirs(dst)
    for f in ("__init__.py", "vfa_oracle.c", "schedule.py"):
        shutil.copy(os.path.join(ROOT, "oracle", f), os.path.join(dst, f))
    if mutation:
        _, old, new = mutation
        src = os.path.join(dst, "vfa_oracle.c")
        text = open(src).read()
        assert text.count(old) == 1, f"mutation anchor not found once: {old!r}"
        open(src, "w").write(text.replace(old, new))


def _run_checks(tmp_path):
    r = subprocess.run([sys.executable, "-c", CHECKS, str(tmp_path), ROOT], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_unmutated_copy_passes_every_check(tmp_path):
    _copy_oracle(str(tmp_path / "oracle"))
    res = _run_checks(tmp_path)
    bad = {k: v for k, v in res.items() if not v <= TOL}
    assert not bad, bad


@pytest.mark.parametrize("mutation", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(tmp_path, mutation):
    _copy_oracle(str(tmp_path / "oracle"), mutation)
    res = _run_checks(tmp_path)
    caught = {k: v for k, v in res.items() if not v <= TOL}
    assert caught, f"{mutation[0]} passed every check: {res}"
