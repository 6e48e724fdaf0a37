"""Host-side checks of libvfa (no GPU): it builds, loads, exports every symbol
that include/vfa.h declares, and rejects bad arguments before touching a
device.  No call here launches a kernel."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def vfa():
    from variable_length_flashattention_gb300 import build, vfa as binding
    build.build()
    binding.lib()
    return binding


def _declared_symbols():
    with open(os.path.join(ROOT, "include", "vfa.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set(re.findall(r"\b(vfa_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(vfa):
    declared = _declared_symbols()
    assert len(declared) >= 10
    L = vfa.lib()
    for name in declared:
        assert hasattr(L, name), f"{name} declared in vfa.h but not exported"
    bound = {n for n, _, _ in vfa.SIGNATURES}
    assert bound == set(declared), "binding and header disagree"


def test_version_and_tile_shape(vfa):
    assert "sm_103a" in vfa.version()
    assert vfa.tile_shape(64) == (128, 128, True)
    assert vfa.tile_shape(128) == (128, 128, True)
    assert vfa.tile_shape(256) == (128, 64, False)
    with pytest.raises(vfa.VfaError) as e:
        vfa.tile_shape(96)
    assert e.value.status == vfa.VFA_ERR_UNSUPPORTED


def test_workspace_bound_covers_worst_case(vfa):
    # one item per (q tile, head); the bound must hold for any split of total_q
    import oracle
    from variable_length_flashattention_gb300 import workloads as W
    for lengths in ([1] * 50, [129] * 7, [128, 1, 0, 255, 3], [5000]):
        cu = W.cu_seqlens(lengths)
        n_items = len(oracle.schedule(cu, cu, 3, 128, 128, True))
        total = int(cu[-1])
        ws = vfa.workspace_bytes(len(lengths), total, total, 3, 128)
        assert ws >= 256 + 32 * n_items
    assert vfa.lib().vfa_varlen_fwd_workspace_bytes(0, 10, 10, 1, 128) == 0
    assert vfa.lib().vfa_varlen_fwd_workspace_bytes(1, 10, 10, 1, 80) == 0


def test_host_rejects_null_and_unsupported(vfa):
    L = vfa.lib()
    nul = None
    st = L.vfa_varlen_fwd(nul, nul, nul, nul, nul, 1, 1, 1, 1, 1, 1, 128, 1.0, 0, -1, nul, nul, nul, 0,
                          nul)
    assert st == vfa.VFA_ERR_INVALID_ARG
    assert b"null" in L.vfa_last_error()
    fake = ctypes.c_void_p(0x100000)   # never dereferenced: rejected before any device work
    st = L.vfa_varlen_fwd(fake, fake, fake, fake, fake, 1, 1, 1, 1, 1, 1, 96, 1.0, 0, -1, fake, fake,
                          fake, 1 << 20, nul)
    assert st == vfa.VFA_ERR_UNSUPPORTED
    st = L.vfa_varlen_fwd(fake, fake, fake, fake, fake, 1, 1, 1, 1, 1, 1, 128, 1.0, 0, -1, fake, fake,
                          fake, 16, nul)
    assert st == vfa.VFA_ERR_INVALID_ARG and b"workspace too small" in L.vfa_last_error()
    st = L.vfa_varlen_fwd(fake, fake, fake, fake, fake, 1, 1, 1, 1, 6, 4, 128, 1.0, 0, -1, fake, fake,
                          fake, 1 << 20, nul)
    assert st == vfa.VFA_ERR_INVALID_ARG and b"num_kv_heads" in L.vfa_last_error()
    odd = ctypes.c_void_p(0x100002)
    st = L.vfa_varlen_fwd(odd, fake, fake, fake, fake, 1, 1, 1, 1, 1, 1, 128, 1.0, 0, -1, fake, fake,
                          fake, 1 << 20, nul)
    assert st == vfa.VFA_ERR_INVALID_ARG and b"aligned" in L.vfa_last_error()
    # a sliding window without a causal mode
    st = L.vfa_varlen_fwd(fake, fake, fake, fake, fake, 1, 1, 1, 1, 1, 1, 128, 1.0, 0, 16, fake, fake,
                          fake, 1 << 20, nul)
    assert st == vfa.VFA_ERR_INVALID_ARG and b"window" in L.vfa_last_error()
    # decode: unsupported group size / block size / head_dim
    st = L.vfa_paged_decode_step(fake, fake, fake, 4, fake, fake, nul, 2, 1, 12, 4, 128, 16, 0.0,
                                 fake, fake, fake, nul, nul)
    assert st == vfa.VFA_ERR_UNSUPPORTED
    st = L.vfa_paged_decode_step(fake, fake, fake, 4, fake, fake, nul, 2, 1, 8, 2, 128, 32, 0.0,
                                 fake, fake, fake, nul, nul)
    assert st == vfa.VFA_ERR_UNSUPPORTED
    st = L.vfa_paged_decode_step(fake, fake, fake, 4, fake, fake, nul, 2, 1, 9, 2, 128, 16, 0.0,
                                 fake, fake, fake, nul, nul)
    assert st == vfa.VFA_ERR_INVALID_ARG
    st = L.vfa_paged_decode_step(fake, fake, fake, 4, fake, fake, nul, 2, 1, 8, 2, 128, 16,
                                 float("nan"), fake, fake, fake, nul, nul)
    assert st == vfa.VFA_ERR_INVALID_ARG and b"softmax_scale" in L.vfa_last_error()
    st = L.vfa_paged_decode_finalize(fake, fake, 1, 1, 12, fake, nul)
    assert st == vfa.VFA_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(vfa):
    import torch
    x = torch.zeros(4, 1, 64, dtype=torch.bfloat16)
    cu = torch.tensor([0, 4], dtype=torch.int32)
    with pytest.raises(ValueError):
        vfa.varlen_fwd(x, x, x, cu, cu, 4, 0.125, False)


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "variable_length_flashattention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                with open(os.path.join(dirpath, fn)) as f:
                    src = f.read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), fn
                assert "vfa_oracle" not in src, fn


def test_backward_and_fp8_host_checks(vfa):
    # rejected on the host before any device work (no GPU needed)
    L = vfa.lib()
    fake = ctypes.c_void_p(0x100000)
    nul = None
    args = lambda D, scale, causal, wl, q=fake: (q, fake, fake, fake, fake, fake, fake, fake,
                                                 4, 4, 1, 2, 2, D, scale, causal, wl, fake, fake,
                                                 fake, fake, 1 << 30, nul)
    assert L.vfa_varlen_bwd(*args(128, 0.1, 1, -1, q=nul)) == vfa.VFA_ERR_INVALID_ARG
    assert b"null" in L.vfa_last_error()
    assert L.vfa_varlen_bwd(*args(96, 0.1, 1, -1)) == vfa.VFA_ERR_UNSUPPORTED
    assert L.vfa_varlen_bwd(*args(128, 0.0, 1, -1)) == vfa.VFA_ERR_INVALID_ARG
    assert L.vfa_varlen_bwd(*args(128, 0.1, 0, 8)) == vfa.VFA_ERR_INVALID_ARG
    assert b"window" in L.vfa_last_error()
    assert L.vfa_varlen_bwd(*args(128, 0.1, 3, -1)) == vfa.VFA_ERR_INVALID_ARG
    assert L.vfa_varlen_bwd_workspace_bytes(1, 10, 2, 96) == 0
    assert L.vfa_varlen_bwd_workspace_bytes(1, 10, 2, 256) > 0
    # status word, key-tile and q-tile starts, Delta; no fp32 dq sum (dq is
    # accumulated in TMEM per query tile)
    assert L.vfa_varlen_bwd_workspace_bytes(2, 10, 2, 128) >= 256 + 2 * 3 * 4 + 10 * 2 * 4
    assert L.vfa_varlen_bwd_workspace_bytes(2, 10, 2, 128) < 10 * 2 * 128 * 4
    # FP8 forward: head_dim 64, 128 or 256, descales finite and positive
    f8 = lambda D, dq, dk: (fake, fake, fake, fake, fake, 4, 4, 4, 1, 2, 2, D, 0.1, dq, dk, 1, -1,
                            fake, fake, fake, 1 << 30, nul)
    assert L.vfa_varlen_fwd_fp8(*f8(96, 1.0, 1.0)) == vfa.VFA_ERR_UNSUPPORTED
    assert L.vfa_varlen_fwd_fp8(*f8(128, 0.0, 1.0)) == vfa.VFA_ERR_INVALID_ARG
    assert L.vfa_varlen_fwd_fp8(*f8(128, 1.0, float("inf"))) == vfa.VFA_ERR_INVALID_ARG


def test_noalloc_rejects_problems_beyond_the_static_scratch(vfa):
    # The static scratch of vfa_varlen_fwd_noalloc holds 1 MiB; a problem whose
    # workspace is larger is refused on the host, before any device work.
    L = vfa.lib()
    nul = None
    # 100k one-token sequences x 8 heads need far more than 1 MiB of work list
    assert L.vfa_varlen_fwd_workspace_bytes(100000, 100000, 100000, 8, 128) > (1 << 20)
    st = L.vfa_varlen_fwd_noalloc(nul, nul, nul, nul, nul, 100000, 100000, 1, 100000, 8, 8, 128,
                                  0.1, 0, -1, nul, nul, nul, nul)
    assert st == vfa.VFA_ERR_UNSUPPORTED
    assert b"static scratch" in L.vfa_last_error()
    # the limit is the exact size: one work item (32 bytes) past it is refused
    r = lambda x: (x + 255) // 256 * 256
    size = lambda B, tq, H: r(r(256 + 32 * H * (tq // 128 + B)) + 56 * (B + 1))
    B, H = 1, 1
    tq = 128 * ((1 << 20) - 1024) // 32         # just inside
    while size(B, tq + 128, H) <= (1 << 20):
        tq += 128
    assert size(B, tq, H) <= (1 << 20) < size(B, tq + 128, H)
    assert L.vfa_varlen_fwd_workspace_bytes(B, tq, tq, H, 128) == size(B, tq, H)
    st = L.vfa_varlen_fwd_noalloc(nul, nul, nul, nul, nul, tq + 128, tq + 128, 1, B, H, H, 128,
                                  0.1, 0, -1, nul, nul, nul, nul)
    assert st == vfa.VFA_ERR_UNSUPPORTED
    # within the limit the call gets past the size check (and then stops at the
    # missing device or the null pointers)
    st = L.vfa_varlen_fwd_noalloc(nul, nul, nul, nul, nul, tq, tq, 1, B, H, H, 128, 0.1, 0, -1,
                                  nul, nul, nul, nul)
    assert st in (vfa.VFA_ERR_INVALID_ARG, vfa.VFA_ERR_CUDA)
    assert b"static scratch" not in L.vfa_last_error()


def test_split_decode_host_checks(vfa):
    # the split step's workspace size is exact and its arguments are checked
    # on the host before any device work (no GPU needed)
    L = vfa.lib()
    r = lambda x: (x + 255) // 256 * 256
    for S, Hq, Hkv, D, n in ((4, 32, 8, 128, 19), (1, 8, 8, 64, 1), (64, 32, 8, 256, 1024)):
        want = r(r(S * Hkv * 4) + S * Hq * n * (D + 2) * 4)
        assert L.vfa_paged_decode_split_workspace_bytes(S, Hq, Hkv, D, n) == want
    # unsupported sizes give 0
    assert L.vfa_paged_decode_split_workspace_bytes(4, 32, 8, 96, 4) == 0       # head_dim
    assert L.vfa_paged_decode_split_workspace_bytes(4, 30, 8, 128, 4) == 0      # Hq % Hkv
    assert L.vfa_paged_decode_split_workspace_bytes(4, 32, 8, 128, 0) == 0      # runs
    assert L.vfa_paged_decode_split_workspace_bytes(4, 32, 8, 128, 1025) == 0
    assert L.vfa_paged_decode_split_workspace_bytes(0, 32, 8, 128, 4) == 0
    # run count: null result pointer and bad sizes
    n = ctypes.c_int(0)
    assert L.vfa_paged_decode_split_count(4, 8, 32, None) == vfa.VFA_ERR_INVALID_ARG
    assert L.vfa_paged_decode_split_count(0, 8, 32, ctypes.byref(n)) == vfa.VFA_ERR_INVALID_ARG
    assert L.vfa_paged_decode_split_count(4, 0, 32, ctypes.byref(n)) == vfa.VFA_ERR_INVALID_ARG
    # split step: run count outside [1, 1024], missing or misaligned workspace,
    # too small a workspace
    fake = ctypes.c_void_p(0x100000)
    ws = ctypes.c_void_p(0x200000)
    step = lambda splits, w, wbytes: L.vfa_paged_decode_step_split(
        fake, fake, fake, 64, fake, fake, None, 32, 4, 32, 8, 128, 16, 0.1, fake, fake, fake,
        None, splits, w, wbytes, None)
    assert step(0, ws, 1 << 30) == vfa.VFA_ERR_INVALID_ARG
    assert step(1025, ws, 1 << 30) == vfa.VFA_ERR_INVALID_ARG
    assert b"num_splits" in L.vfa_last_error()
    assert step(4, None, 1 << 30) == vfa.VFA_ERR_INVALID_ARG
    assert step(4, ctypes.c_void_p(0x200010), 1 << 30) == vfa.VFA_ERR_INVALID_ARG
    need = L.vfa_paged_decode_split_workspace_bytes(4, 32, 8, 128, 4)
    assert step(4, ws, need - 1) == vfa.VFA_ERR_INVALID_ARG
    assert b"too small" in L.vfa_last_error()
