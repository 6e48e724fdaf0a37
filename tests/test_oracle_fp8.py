"""Pins for the FP8 (E4M3 q and k) forward oracle (CPU only).

  * the E4M3 decoder against torch's float8_e4m3fn conversion for all 256
    codes, and hand-decoded values of the format's definition;
  * the FP8 forward against torch float64 scaled_dot_product_attention on
    torch-decoded q and k;
  * codes whose values bf16 holds exactly (descale a power of two) give the
    bf16 forward's result bit for bit.
"""
import numpy as np
import pytest
import torch

from variable_length_flashattention_gb300 import workloads as W


def test_decoder_matches_torch_for_every_code(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle_mod.fp8_e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[ok], ref[ok])


def test_decoder_hand_values(oracle_mod):
    # 0 0111 000 = 1.0; 0 0000 001 = 2^-9 (smallest subnormal); 0 0001 000 = 2^-6;
    # 0 1111 110 = 448 (largest); 1 0111 100 = -1.5; 0 1111 111 = NaN
    codes = np.array([0x38, 0x01, 0x08, 0x7E, 0xBC, 0x7F], dtype=np.uint8)
    got = oracle_mod.fp8_e4m3_decode(codes)
    np.testing.assert_array_equal(got[:5], [1.0, 2.0 ** -9, 2.0 ** -6, 448.0, -1.5])
    assert np.isnan(got[5])


def _dequant(codes, descale):
    return codes.view(torch.float8_e4m3fn).to(torch.float64) * descale


@pytest.mark.parametrize("causal,window_left", [(0, -1), (1, -1), (2, -1), (1, 30)])
def test_matches_torch_sdpa_float64(oracle_mod, causal, window_left):
    lq, lk = [5, 90, 1, 0, 40], [9, 90, 4, 6, 70]
    H, D = 2, 32
    case = W.make_varlen("fp8", lq, lk, H, D, bool(causal), 1.0, value_seed=3 + causal)
    f8 = W.fp8_qk(case)
    out, lse, _ = oracle_mod.varlen_fwd_fp8(f8.q8, f8.k8, case.v, case.cu_seqlens_q,
                                            case.cu_seqlens_k, H, D, case.softmax_scale,
                                            f8.descale_q, f8.descale_k, causal,
                                            window_left=window_left)
    q = _dequant(f8.q8, f8.descale_q)
    k = _dequant(f8.k8, f8.descale_k)
    v = case.v.double()
    for b in range(case.batch):
        q0, q1 = int(case.cu_seqlens_q[b]), int(case.cu_seqlens_q[b + 1])
        k0, k1 = int(case.cu_seqlens_k[b]), int(case.cu_seqlens_k[b + 1])
        if q1 == q0 or k1 == k0:
            continue
        off = (k1 - k0) - (q1 - q0) if causal == 2 else 0
        i = torch.arange(q1 - q0)[:, None]
        j = torch.arange(k1 - k0)[None, :]
        allowed = torch.ones(q1 - q0, k1 - k0, dtype=torch.bool)
        if causal:
            allowed &= j <= i + off
        if window_left >= 0:
            allowed &= j >= i + off - window_left
        live = allowed.any(dim=1)
        qs = q[q0:q1].transpose(0, 1)[:, live]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qs, k[k0:k1].transpose(0, 1), v[k0:k1].transpose(0, 1), attn_mask=allowed[live],
            scale=case.softmax_scale)
        np.testing.assert_allclose(out[q0:q1][live.numpy()], ref.transpose(0, 1).numpy(),
                                   rtol=1e-10, atol=1e-12)


def test_equals_bf16_forward_on_exact_values(oracle_mod):
    lq, lk = [70, 3, 129], [70, 50, 129]
    case = W.make_varlen("fp8-exact", lq, lk, 2, 64, True, 1.0, value_seed=9)
    f8 = W.fp8_qk(case)
    o8, l8, _ = oracle_mod.varlen_fwd_fp8(f8.q8, f8.k8, case.v, case.cu_seqlens_q,
                                          case.cu_seqlens_k, 2, 64, case.softmax_scale,
                                          f8.descale_q, f8.descale_k, True)
    qb = _dequant(f8.q8, f8.descale_q).to(torch.bfloat16)
    kb = _dequant(f8.k8, f8.descale_k).to(torch.bfloat16)
    assert torch.equal(qb.double(), _dequant(f8.q8, f8.descale_q))   # exact in bf16
    ob, lb, _ = oracle_mod.varlen_fwd(qb, kb, case.v, case.cu_seqlens_q, case.cu_seqlens_k, 2, 64,
                                      case.softmax_scale, True)
    np.testing.assert_array_equal(o8, ob)
    np.testing.assert_array_equal(l8, lb)
