"""vfa_varlen_fwd_noalloc: the varlen forward for callers that cannot allocate
device memory (its scratch is a fixed array inside the library).

It must give the same results as vfa_varlen_fwd, whose caller supplies the
workspace, on two calls in a row (the second call runs on the scratch the
first one left behind).  This file is collected last on purpose: it shares
the library's static scratch, and it must pass both on its own in a fresh
process and after every other test.
"""
import numpy as np
import pytest
import torch

from helpers import LSE_ATOL, OUT_ATOL, OUT_RTOL
from variable_length_flashattention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vfa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from variable_length_flashattention_gb300 import build, vfa as binding
    build.build()
    return binding


def _close(a_out, a_lse, b_out, b_lse):
    a = a_out.float().cpu().double().numpy()
    b = b_out.float().cpu().double().numpy()
    assert np.all(np.isfinite(a))
    assert np.all(np.abs(a - b) <= OUT_ATOL + OUT_RTOL * np.abs(b))
    la, lb = a_lse.cpu().double().numpy(), b_lse.cpu().double().numpy()
    assert np.all(np.abs(la - lb) <= LSE_ATOL)


@pytest.mark.parametrize("name", ["tiny-causal", "packed", "cross-d64"])
def test_noalloc_matches_workspace_entry_twice(vfa, name):
    case = W.VARLEN_WORKLOADS[name](0)
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    cq = torch.from_numpy(case.cu_seqlens_q).cuda()
    ck = torch.from_numpy(case.cu_seqlens_k).cuda()
    ref_out, ref_lse = vfa.varlen_fwd(q, k, v, cq, ck, case.max_seqlen_q, case.softmax_scale,
                                      case.causal)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((case.total_q, case.num_heads), float("nan"), device="cuda")
        vfa.varlen_fwd_noalloc(q, k, v, cq, ck, case.max_seqlen_q, case.softmax_scale,
                               case.causal, out, lse, device_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        _close(out, lse, ref_out, ref_lse)


def test_noalloc_rejects_problems_beyond_the_static_scratch(vfa):
    # 100k one-token sequences x 8 heads need far more than 1 MiB of work list
    L = vfa.lib()
    fake = None
    st = L.vfa_varlen_fwd_noalloc(fake, fake, fake, fake, fake, 100000, 100000, 1, 100000, 8,
                                  8, 128, 0.1, 0, -1, fake, fake, fake, None)
    assert st == vfa.VFA_ERR_UNSUPPORTED
    assert b"static scratch" in L.vfa_last_error()
