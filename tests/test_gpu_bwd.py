"""GPU parity of vfa_varlen_bwd against the fp64 backward oracle (through the C ABI).

The forward's out and lse come from the GPU forward, as in training.  P and
dS are rounded to bf16 for the tensor-core products and the gradients to bf16
at the end, so each gradient element is held to the first-order bound of
those roundings (tests/bwd_error_model.py):
    |got - ref| <= 2 * 2^-8 * (|ref| + M) + 1e-6
where M sums the absolute values of the terms the rounded quantities enter
(for dV: sum_i P_ij |dO_i|).  Outputs start as NaN canaries.
"""
import numpy as np
import pytest
import torch

from bwd_error_model import check_grad, magnitudes
from helpers import to_dev
from variable_length_flashattention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module")
def vfa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from variable_length_flashattention_gb300 import build, vfa as binding
    build.build()
    return binding


def _nan_like(t):
    return torch.full_like(t.view(torch.int16), 0x7FC0).view(torch.bfloat16)


def _run(vfa, case, dout, causal, window_left=-1):
    d = to_dev(case)
    out, lse = vfa.varlen_fwd(d["q"], d["k"], d["v"], d["cu_q"], d["cu_k"], case.max_seqlen_q,
                              case.softmax_scale, causal, window_left=window_left)
    g = dout.cuda()
    dq, dk, dv = _nan_like(d["q"]), _nan_like(d["k"]), _nan_like(d["v"])
    _, _, _, ws = vfa.varlen_bwd(d["q"], d["k"], d["v"], out, g, lse, d["cu_q"], d["cu_k"],
                                 case.softmax_scale, causal, window_left, dq=dq, dk=dk, dv=dv)
    status = vfa.read_status(ws)
    torch.cuda.synchronize()
    f = lambda t: t.float().cpu().double().numpy()
    return f(dq), f(dk), f(dv), status


def _check(got, ref, mag, what):
    check_grad(got, ref, mag, what)


def _compare(vfa, oracle_mod, case, causal, window_left=-1, Hkv=None, seed=0):
    dout = W.upstream_grad(case, seed)
    dq, dk, dv, status = _run(vfa, case, dout, causal, window_left)
    assert status == 0
    H, D = case.num_heads, case.head_dim
    rq, rk, rv, _ = oracle_mod.varlen_bwd(case.q, case.k, case.v, dout, case.cu_seqlens_q,
                                          case.cu_seqlens_k, H, D, case.softmax_scale, causal,
                                          num_kv_heads=Hkv or H, window_left=window_left)
    mq, mk, mv = magnitudes(case, dout, causal, window_left, Hkv or H)
    what = f"{case.name} causal {causal} window {window_left} D={D} H={H}/{Hkv or H}"
    _check(dq, rq, mq, "dq " + what)
    _check(dk, rk, mk, "dk " + what)
    _check(dv, rv, mv, "dv " + what)


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("causal", [0, 1])
def test_tiny(vfa, oracle_mod, causal, seed):
    _compare(vfa, oracle_mod, W.tiny(bool(causal), seed), causal, seed=seed)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [0, 1, 2])
def test_small_mixes(vfa, oracle_mod, D, causal):
    lq = [1, 7, 64, 129, 300, 0, 257]
    lk = [1, 7, 64, 129, 300, 5, 90] if causal == 2 else [1, 7, 64, 129, 300, 5, 257]
    case = W.make_varlen("bwd", lq, lk, 2, D, bool(causal), 1.0, value_seed=D + causal)
    _compare(vfa, oracle_mod, case, causal, seed=causal)


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("window_left", [0, 100, 300])
@pytest.mark.parametrize("causal", [1, 2])
def test_sliding_window(vfa, oracle_mod, window_left, causal, D):
    lq, lk = [500, 64, 700, 1], [500, 300, 400, 50]
    case = W.make_varlen("bwd-window", lq, lk, 2, D, True, 1.0, value_seed=7 + window_left)
    _compare(vfa, oracle_mod, case, causal, window_left=window_left, seed=window_left)


@pytest.mark.parametrize("H,Hkv,D", [(8, 2, 128), (4, 1, 64), (4, 2, 256)])
def test_grouped_kv_heads(vfa, oracle_mod, H, Hkv, D):
    lq, lk = [300, 7, 129, 64], [300, 40, 129, 200]
    case = W.make_varlen("bwd-gqa", lq, lk, H, D, True, 1.0, value_seed=H + Hkv)
    case.k = case.k[:, :Hkv].contiguous()
    case.v = case.v[:, :Hkv].contiguous()
    _compare(vfa, oracle_mod, case, 1, Hkv=Hkv, seed=3)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_packed_batch(vfa, oracle_mod, seed):
    # the packed workload (16 sequences up to 2048 tokens, H=16, D=128,
    # causal), every sequence and head, in the launch configuration the
    # bench times
    _compare(vfa, oracle_mod, W.packed(seed), 1, seed=seed)


def test_bad_cu_seqlens_sets_status(vfa):
    case = W.make_varlen("bad", [10, 20], [10, 20], 1, 64, True, 1.0, value_seed=1)
    d = to_dev(case)
    out, lse = vfa.varlen_fwd(d["q"], d["k"], d["v"], d["cu_q"], d["cu_k"], 20,
                              case.softmax_scale, True)
    bad = d["cu_q"].clone()
    bad[1] = 35                                  # [0, 35, 30]: decreasing
    dq = _nan_like(d["q"])
    _, _, _, ws = vfa.varlen_bwd(d["q"], d["k"], d["v"], out, out, lse, bad, d["cu_k"],
                                 case.softmax_scale, 1, dq=dq)
    assert vfa.read_status(ws) == vfa.VFA_ERR_BAD_SEQLENS
    assert torch.isnan(dq.float()).all()


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [0, 1, 2])
def test_step_boundaries(vfa, oracle_mod, causal, D):
    # The dQ kernel streams keys in steps of 96, the dK/dV kernel queries in
    # steps of 96 at head_dim 64 (64 at 128): lengths at, just below and just
    # above multiples of 96 (and of the 128-row tiles) end steps at every
    # offset, with the next sequence's rows right behind the last step.
    lq = [95, 96, 97, 191, 192, 193, 288, 64]
    lk = [95, 96, 97, 191, 192, 193, 288, 300] if causal == 2 else lq
    case = W.make_varlen("bwd-steps", lq, lk, 2, D, bool(causal), 1.0, value_seed=60 + D + causal)
    _compare(vfa, oracle_mod, case, causal, seed=60 + causal)


@pytest.mark.parametrize("D", [64, 256])
@pytest.mark.parametrize("causal", [0, 1, 2])
def test_edge_lengths(vfa, oracle_mod, causal, D):
    # a query sequence with no keys (dq = 0), keys no query sees (dk = dv = 0),
    # one-token sequences and an empty sequence between non-empty ones
    lq = [10, 0, 1, 130, 3]
    lk = [0, 7, 1, 130, 200]
    case = W.make_varlen("bwd-edge", lq, lk, 2, D, bool(causal), 1.0, value_seed=40 + causal)
    _compare(vfa, oracle_mod, case, causal, seed=40)


def test_deterministic(vfa):
    # no gradient is accumulated with atomics: two runs agree bit for bit
    case = W.packed(2)
    dout = W.upstream_grad(case, 2)
    a = _run(vfa, case, dout, 1)
    b = _run(vfa, case, dout, 1)
    for x, y in zip(a[:3], b[:3]):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_cross_attention_d256(vfa, oracle_mod, seed):
    # the cross-attention workload at head_dim 256 (32 sequences, q up to 512,
    # k up to 4096 tokens, non-causal), every sequence and head
    _compare(vfa, oracle_mod, W.cross(256, seed), 0, seed=seed)


def test_longtail_longest_sequences(vfa, oracle_mod):
    # the long-tail workload's 8192-token sequence (H=32, sigma 0.5) with two
    # of its short sequences: long units of the persistent kernels, many
    # query blocks per key tile, every element against the oracle
    full = W.longtail(0)
    L = full.lengths_q
    picks = [L.index(8192)] + [i for i in range(len(L)) if L[i] < 300][:2]
    lens = [L[i] for i in picks]
    case = W.make_varlen("longtail-sub", lens, lens, 32, 128, True, 0.5, value_seed=0)
    parts_q, parts_k, parts_v = [], [], []
    for i in picks:
        r0, r1 = int(full.cu_seqlens_q[i]), int(full.cu_seqlens_q[i + 1])
        parts_q.append(full.q[r0:r1])
        parts_k.append(full.k[r0:r1])
        parts_v.append(full.v[r0:r1])
    case.q = torch.cat(parts_q).contiguous()
    case.k = torch.cat(parts_k).contiguous()
    case.v = torch.cat(parts_v).contiguous()
    _compare(vfa, oracle_mod, case, 1, seed=0)
