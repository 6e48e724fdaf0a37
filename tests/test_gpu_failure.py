"""Failure detection without a GPU fault: a wait that nothing satisfies must
give up after the bounded-wait limit, report VFA_ERR_TIMEOUT through the
status word, and leave the context usable for the next call."""
import time

import pytest
import torch

from helpers import assert_lse_close, assert_out_close, run_varlen
from variable_length_flashattention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vfa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from variable_length_flashattention_gb300 import build, vfa as binding
    build.build()
    return binding


def test_bounded_wait_times_out_and_context_stays_usable(vfa, oracle_mod):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    vfa.debug_bounded_wait(status)
    st = vfa.read_status(status)
    dt = time.perf_counter() - t0
    assert st == vfa.VFA_ERR_TIMEOUT
    assert 0.5 < dt < 60.0                         # the 1 s limit, not an endless spin
    case = W.tiny(True, 0)                         # the next call runs normally
    out, lse, s2 = run_varlen(vfa, case)
    assert s2 == 0
    ref_out, ref_lse, _ = oracle_mod.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens_q,
                                                case.cu_seqlens_k, case.num_heads,
                                                case.head_dim, case.softmax_scale, True)
    assert_out_close(out, ref_out, "after timeout")
    assert_lse_close(lse, ref_lse, "after timeout")
