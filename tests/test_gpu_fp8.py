"""GPU parity of vfa_varlen_fwd_fp8 (FP8 E4M3 q and k, bf16 v) against the fp64 oracle.

The tensor core's FP8 products are exact and accumulate in fp32, as the
bf16 products do, so the forward's tolerances apply unchanged (helpers.py).
"""
import numpy as np
import pytest
import torch

from helpers import BF16_NAN, assert_lse_close, assert_out_close
from variable_length_flashattention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vfa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from variable_length_flashattention_gb300 import build, vfa as binding
    build.build()
    return binding


def _run(vfa, case, f8, causal, window_left=-1):
    q8, k8, v = f8.q8.cuda(), f8.k8.cuda(), case.v.cuda()
    cq = torch.from_numpy(case.cu_seqlens_q).cuda()
    ck = torch.from_numpy(case.cu_seqlens_k).cuda()
    out = torch.full(case.q.shape, 0, dtype=torch.int16, device="cuda").fill_(BF16_NAN)
    out = out.view(torch.bfloat16)
    lse = torch.full((case.total_q, case.num_heads), float("nan"), device="cuda")
    ws = vfa.alloc_workspace(case.batch, case.total_q, case.total_k, case.num_heads,
                             case.head_dim)
    vfa.varlen_fwd_fp8(q8, k8, v, cq, ck, max(case.max_seqlen_q, 0), case.softmax_scale,
                       f8.descale_q, f8.descale_k, causal, out=out, lse=lse, workspace=ws,
                       window_left=window_left)
    status = vfa.read_status(ws)
    torch.cuda.synchronize()
    return out.float().cpu().double().numpy(), lse.cpu().double().numpy(), status


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal,window_left", [(0, -1), (1, -1), (2, -1), (1, 200), (2, 37)])
def test_mixes(vfa, oracle_mod, causal, window_left, D):
    lq = [1, 7, 64, 129, 300, 0, 257, 1000]
    lk = [1, 7, 64, 129, 300, 5, 90, 800]
    case = W.make_varlen("fp8", lq, lk, 2, D, bool(causal), 1.0, value_seed=20 + causal + D)
    f8 = W.fp8_qk(case)
    out, lse, status = _run(vfa, case, f8, causal, window_left)
    assert status == 0
    ref_out, ref_lse, _ = oracle_mod.varlen_fwd_fp8(f8.q8, f8.k8, case.v, case.cu_seqlens_q,
                                                    case.cu_seqlens_k, 2, D,
                                                    case.softmax_scale, f8.descale_q,
                                                    f8.descale_k, causal,
                                                    window_left=window_left)
    assert_out_close(out, ref_out, f"fp8 D={D} causal {causal} window {window_left}")
    assert_lse_close(lse, ref_lse, f"fp8 D={D} causal {causal} window {window_left}")


@pytest.mark.parametrize("D", [64, 128, 256])
def test_grouped_kv_heads(vfa, oracle_mod, D):
    lq, lk = [300, 7, 129, 64], [300, 40, 129, 200]
    case = W.make_varlen("fp8-gqa", lq, lk, 8, D, True, 1.0, value_seed=31 + D)
    case.k = case.k[:, :2].contiguous()
    case.v = case.v[:, :2].contiguous()
    f8 = W.fp8_qk(case)
    out, lse, status = _run(vfa, case, f8, 1)
    assert status == 0
    ref_out, ref_lse, _ = oracle_mod.varlen_fwd_fp8(f8.q8, f8.k8, case.v, case.cu_seqlens_q,
                                                    case.cu_seqlens_k, 8, D,
                                                    case.softmax_scale, f8.descale_q,
                                                    f8.descale_k, 1, num_kv_heads=2)
    assert_out_close(out, ref_out, "fp8 gqa")
    assert_lse_close(lse, ref_lse, "fp8 gqa")


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_packed_batch(vfa, oracle_mod, seed):
    # the bench's packed batch with FP8 q and k, every sequence and head
    case = W.packed(seed)
    f8 = W.fp8_qk(case)
    out, lse, status = _run(vfa, case, f8, 1)
    assert status == 0
    ro, rl, _ = oracle_mod.varlen_fwd_fp8(f8.q8, f8.k8, case.v, case.cu_seqlens_q,
                                          case.cu_seqlens_k, 16, 128, case.softmax_scale,
                                          f8.descale_q, f8.descale_k, 1)
    assert_out_close(out, ro, f"fp8 packed seed {seed}")
    assert_lse_close(lse, rl, f"fp8 packed seed {seed}")


@pytest.mark.parametrize("seed", [0, 1])
def test_cross_attention_d256(vfa, oracle_mod, seed):
    # the cross-attention workload at head_dim 256 with FP8 q and k
    case = W.cross(256, seed)
    f8 = W.fp8_qk(case)
    out, lse, status = _run(vfa, case, f8, 0)
    assert status == 0
    ro, rl, _ = oracle_mod.varlen_fwd_fp8(f8.q8, f8.k8, case.v, case.cu_seqlens_q,
                                          case.cu_seqlens_k, 8, 256, case.softmax_scale,
                                          f8.descale_q, f8.descale_k, 0)
    assert_out_close(out, ro, f"fp8 cross-d256 seed {seed}")
    assert_lse_close(lse, rl, f"fp8 cross-d256 seed {seed}")


def test_rejects_other_head_dims_and_bad_descales(vfa):
    case = W.make_varlen("fp8-d96", [8], [8], 1, 96, True, 1.0, value_seed=1)
    f8 = W.fp8_qk(case)
    with pytest.raises(vfa.VfaError):
        _run(vfa, case, f8, 1)
    case = W.make_varlen("fp8-bad", [8], [8], 1, 128, True, 1.0, value_seed=1)
    f8 = W.fp8_qk(case)
    f8.descale_q = 0.0
    with pytest.raises(vfa.VfaError):
        _run(vfa, case, f8, 1)


@pytest.mark.parametrize("causal", [0, 1, 2])
def test_edge_lengths(vfa, oracle_mod, causal):
    lq = [10, 0, 1, 130, 3]
    lk = [0, 7, 1, 130, 200]
    case = W.make_varlen("fp8-edge", lq, lk, 2, 128, bool(causal), 1.0, value_seed=50 + causal)
    f8 = W.fp8_qk(case)
    out, lse, status = _run(vfa, case, f8, causal)
    assert status == 0
    ref_out, ref_lse, _ = oracle_mod.varlen_fwd_fp8(f8.q8, f8.k8, case.v, case.cu_seqlens_q,
                                                    case.cu_seqlens_k, 2, 128,
                                                    case.softmax_scale, f8.descale_q,
                                                    f8.descale_k, causal)
    assert_out_close(out, ref_out, f"fp8 edge causal {causal}")
    assert_lse_close(lse, ref_lse, f"fp8 edge causal {causal}")


@pytest.mark.parametrize("seed", [0, 1])
def test_cross_attention_d64(vfa, oracle_mod, seed):
    # the cross-attention workload at head_dim 64 with FP8 q and k (64-byte rows)
    case = W.cross(64, seed)
    f8 = W.fp8_qk(case)
    out, lse, status = _run(vfa, case, f8, 0)
    assert status == 0
    ro, rl, _ = oracle_mod.varlen_fwd_fp8(f8.q8, f8.k8, case.v, case.cu_seqlens_q,
                                          case.cu_seqlens_k, 8, 64, case.softmax_scale,
                                          f8.descale_q, f8.descale_k, 0)
    assert_out_close(out, ro, f"fp8 cross-d64 seed {seed}")
    assert_lse_close(lse, rl, f"fp8 cross-d64 seed {seed}")
