"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI,
compare with the oracle at the stated tolerances."""
import numpy as np
import torch

FLT_MAX = float(np.finfo(np.float32).max)

# |out - ref| <= OUT_ATOL + OUT_RTOL * |ref| elementwise (bf16 output);
# |lse - ref| <= LSE_ATOL where a key set exists; lse == -FLT_MAX bit-exact where none.
OUT_ATOL = 1e-2
OUT_RTOL = 1e-2
LSE_ATOL = 2e-3

BF16_NAN = 0x7FC1          # canary bit pattern for unwritten bf16 outputs


def to_dev(case, device="cuda"):
    return dict(q=case.q.to(device), k=case.k.to(device), v=case.v.to(device),
                cu_q=torch.from_numpy(case.cu_seqlens_q).to(device),
                cu_k=torch.from_numpy(case.cu_seqlens_k).to(device))


def run_varlen(vfa, case, device="cuda", workspace=None, window_left=-1):
    """GPU forward with NaN-canary outputs; returns (out f64 numpy, lse f64 numpy, status)."""
    d = to_dev(case, device)
    out = torch.full_like(d["q"].view(torch.int16), BF16_NAN).view(torch.bfloat16)
    lse = torch.full((case.total_q, case.num_heads), float("nan"), dtype=torch.float32,
                     device=device)
    if workspace is None:
        workspace = vfa.alloc_workspace(case.batch, case.total_q, case.total_k, case.num_heads,
                                        case.head_dim, device=device)
    vfa.varlen_fwd(d["q"], d["k"], d["v"], d["cu_q"], d["cu_k"], max(case.max_seqlen_q, 0),
                   case.softmax_scale, case.causal, out=out, lse=lse, workspace=workspace,
                   window_left=window_left)
    status = vfa.read_status(workspace)
    torch.cuda.synchronize()
    return (out.float().cpu().double().numpy(), lse.cpu().double().numpy(), status)


def assert_out_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite (unwritten?) outputs"
    err = np.abs(got - ref)
    bound = OUT_ATOL + OUT_RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst "
                             f"{(err - bound).max():.3g}; first {idx.tolist()}")


def assert_lse_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    empty = ref == -FLT_MAX
    assert np.all(got[empty] == np.float32(-FLT_MAX)), f"{what}: empty rows must hold -FLT_MAX"
    live = ~empty
    assert np.all(np.isfinite(got[live])), f"{what}: non-finite lse"
    err = np.abs(got[live] - ref[live])
    assert err.size == 0 or err.max() <= LSE_ATOL, f"{what}: lse error {err.max():.3g} > {LSE_ATOL}"
