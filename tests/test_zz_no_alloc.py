"""vfa_varlen_fwd_noalloc: the varlen forward for callers that cannot allocate
device memory (its scratch is a fixed array inside the library).

Each call must agree with the fp64 oracle at the forward's tolerances and
with vfa_varlen_fwd (whose caller supplies the workspace).  The calls run
as a chain of different problems on the one shared array, each problem
twice in a row, so a word the scheduler failed to rewrite would carry the
previous problem's work list or records into the next call.  One problem
has more than 2048 sequences, where the scheduler keeps its per-sequence
records in the static array instead of shared memory.

This file is collected last on purpose: it shares the library's static
scratch, and it must pass both on its own in a fresh process and after every
other test.  (The host-side size limit is checked without a GPU in
test_library_host.py.)
"""
import numpy as np
import pytest
import torch

from helpers import (BF16_NAN, LSE_ATOL, OUT_ATOL, OUT_RTOL, assert_lse_close,
                     assert_out_close)
from variable_length_flashattention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vfa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from variable_length_flashattention_gb300 import build, vfa as binding
    build.build()
    return binding


def _many_short(seed):
    # 2500 sequences of 1..9 tokens: 2501 scheduler records exceed the 2048
    # the scheduler holds in shared memory, so they live in the static array
    rng = np.random.default_rng(seed)
    lengths = rng.integers(1, 10, 2500)
    return W.make_varlen("many-short", lengths, lengths, 2, 64, True, 1.0, value_seed=seed + 77)


CHAIN = [
    ("cross-d64", lambda: W.cross(64, 0)),
    ("tiny-causal", lambda: W.tiny(True, 1)),
    ("many-short", lambda: _many_short(3)),
    ("packed", lambda: W.packed(1)),
    ("tiny", lambda: W.tiny(False, 2)),
    ("cross-d256", lambda: W.cross(256, 1)),
]


def _close(got_out, got_lse, ref_out, ref_lse):
    assert np.all(np.isfinite(got_out))
    assert np.all(np.abs(got_out - ref_out) <= OUT_ATOL + OUT_RTOL * np.abs(ref_out))
    assert np.all(np.abs(got_lse - ref_lse) <= LSE_ATOL)


def test_noalloc_chain_matches_oracle_and_workspace_entry(vfa, oracle_mod):
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for name, make in CHAIN:
        case = make()
        q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
        cq = torch.from_numpy(case.cu_seqlens_q).cuda()
        ck = torch.from_numpy(case.cu_seqlens_k).cuda()
        ref_out, ref_lse, _ = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q,
                                                    case.cu_seqlens_k, case.num_heads,
                                                    case.head_dim, case.softmax_scale,
                                                    case.causal)
        ws_out, ws_lse = vfa.varlen_fwd(q, k, v, cq, ck, case.max_seqlen_q, case.softmax_scale,
                                        case.causal)
        ws_out = ws_out.float().cpu().double().numpy()
        ws_lse = ws_lse.cpu().double().numpy()
        for rep in range(2):
            out = torch.full_like(q.view(torch.int16), BF16_NAN).view(torch.bfloat16)
            lse = torch.full((case.total_q, case.num_heads), float("nan"), device="cuda")
            status.fill_(-1)
            vfa.varlen_fwd_noalloc(q, k, v, cq, ck, case.max_seqlen_q, case.softmax_scale,
                                   case.causal, out, lse, device_status=status)
            torch.cuda.synchronize()
            assert int(status.item()) == 0, f"{name} call {rep}: status {int(status.item())}"
            got = out.float().cpu().double().numpy()
            got_lse = lse.cpu().double().numpy()
            assert_out_close(got, ref_out, f"{name} call {rep} vs oracle")
            assert_lse_close(got_lse, ref_lse, f"{name} call {rep} vs oracle")
            _close(got, got_lse, ws_out, ws_lse)


def test_noalloc_bad_cu_seqlens_reports_status_then_recovers(vfa, oracle_mod):
    # a device-detected error leaves its mark only in this call's status word:
    # the next call on the same static array runs normally
    case = W.tiny(True, 0)
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    cq = torch.from_numpy(case.cu_seqlens_q).cuda()
    ck = torch.from_numpy(case.cu_seqlens_k).cuda()
    bad = cq.clone()
    bad[2] = bad[1] - 1
    out = torch.full_like(q, 7.0)
    lse = torch.full((case.total_q, 2), 7.0, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    vfa.varlen_fwd_noalloc(q, k, v, bad, ck, case.max_seqlen_q, case.softmax_scale, True, out,
                           lse, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == vfa.VFA_ERR_BAD_SEQLENS
    assert torch.all(out == 7.0) and torch.all(lse == 7.0)
    vfa.varlen_fwd_noalloc(q, k, v, cq, ck, case.max_seqlen_q, case.softmax_scale, True, out,
                           lse, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_out, ref_lse, _ = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q,
                                                case.cu_seqlens_k, 2, 64, case.softmax_scale, True)
    assert_out_close(out.float().cpu().double().numpy(), ref_out, "after a bad call")
    assert_lse_close(lse.cpu().double().numpy(), ref_lse, "after a bad call")
