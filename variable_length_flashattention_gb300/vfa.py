"""Python binding of libvfa (include/vfa.h): argument marshalling only.

Every function takes torch tensors that already live on the current CUDA
device, passes their data pointers and the current torch stream to the C ABI,
and raises ``VfaError`` on a non-OK status.  All computation happens in the
library's kernels; there is no fallback of any kind: if ``libvfa.so`` has not
been built (``python -m variable_length_flashattention_gb300.build``) the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libvfa.so")
_lock = threading.Lock()
_lib = None

STATUS_NAMES = {
    0: "VFA_OK",
    1: "VFA_ERR_INVALID_ARG",
    2: "VFA_ERR_UNSUPPORTED",
    3: "VFA_ERR_ARCH",
    4: "VFA_ERR_CUDA",
    5: "VFA_ERR_BAD_SEQLENS",
    6: "VFA_ERR_BAD_BLOCK",
    7: "VFA_ERR_TIMEOUT",
    8: "VFA_ERR_WORKSPACE",
}
VFA_OK, VFA_ERR_INVALID_ARG, VFA_ERR_UNSUPPORTED, VFA_ERR_ARCH, VFA_ERR_CUDA = 0, 1, 2, 3, 4
VFA_ERR_BAD_SEQLENS, VFA_ERR_BAD_BLOCK, VFA_ERR_TIMEOUT, VFA_ERR_WORKSPACE = 5, 6, 7, 8

# Every symbol include/vfa.h declares: (name, restype, argtypes).
_P, _I, _F, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = [
    ("vfa_last_error", ctypes.c_char_p, []),
    ("vfa_version", ctypes.c_char_p, []),
    ("vfa_varlen_fwd_workspace_bytes", _S, [_I, _I, _I, _I, _I]),
    ("vfa_varlen_fwd_tile_shape", _I, [_I, _P, _P, _P]),
    ("vfa_varlen_fwd", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P, _P, _P,
                            _S, _P]),
    ("vfa_varlen_fwd_fp8", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _F, _F, _I,
                                _I, _P, _P, _P, _S, _P]),
    ("vfa_varlen_fwd_noalloc", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P,
                                    _P, _P, _P]),
    ("vfa_varlen_schedule", _I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _I, _P, _P, _P,
                                 _S, _P]),
    ("vfa_varlen_bwd_workspace_bytes", _S, [_I, _I, _I, _I]),
    ("vfa_varlen_bwd", _I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I,
                            _P, _P, _P, _P, _S, _P]),
    ("vfa_paged_decode_init", _I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    ("vfa_paged_decode_step", _I, [_P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P,
                                   _P, _P, _P, _P]),
    ("vfa_paged_decode_step_split", _I, [_P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F,
                                         _P, _P, _P, _P, _I, _P, _S, _P]),
    ("vfa_paged_decode_split_workspace_bytes", _S, [_I, _I, _I, _I, _I]),
    ("vfa_paged_decode_split_count", _I, [_I, _I, _I, _P]),
    ("vfa_paged_decode_finalize", _I, [_P, _P, _I, _I, _I, _P, _P]),
    ("vfa_debug_paged_gather", _I, [_P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
    ("vfa_debug_bounded_wait", _I, [_P, _P]),
    ("vfa_read_status", _I, [_P, _P, _P]),
]


class VfaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"libvfa.so is not built ({_LIB_PATH}); run "
                "`python -m variable_length_flashattention_gb300.build` first")
        L = ctypes.CDLL(_LIB_PATH)
        for name, res, args in SIGNATURES:
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
        return L


def _check(st: int):
    if st != VFA_OK:
        raise VfaError(st, lib().vfa_last_error().decode(errors="replace"))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def version() -> str:
    return lib().vfa_version().decode()


# ----------------------------------------------------------------- varlen forward

def tile_shape(head_dim: int) -> Tuple[int, int, bool]:
    """(q tile rows, key tile rows, two q tiles per work item) for head_dim."""
    bq, bk, pr = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(lib().vfa_varlen_fwd_tile_shape(head_dim, ctypes.byref(bq), ctypes.byref(bk),
                                           ctypes.byref(pr)))
    return bq.value, bk.value, bool(pr.value)


def workspace_bytes(batch: int, total_q: int, total_k: int, num_heads: int, head_dim: int) -> int:
    n = lib().vfa_varlen_fwd_workspace_bytes(batch, total_q, total_k, num_heads, head_dim)
    if n == 0:
        raise VfaError(VFA_ERR_INVALID_ARG, "no workspace size for these arguments")
    return int(n)


def alloc_workspace(batch: int, total_q: int, total_k: int, num_heads: int, head_dim: int,
                    device=None) -> torch.Tensor:
    n = workspace_bytes(batch, total_q, total_k, num_heads, head_dim)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def varlen_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens_q: torch.Tensor,
               cu_seqlens_k: torch.Tensor, max_seqlen_q: int, softmax_scale: float,
               causal, out: Optional[torch.Tensor] = None,
               lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
               stream=None, window_left: int = -1):
    """out bf16 [Tq, H, D], lse f32 [Tq, H] = varlen attention forward (vfa_varlen_fwd).

    k, v may hold fewer heads than q (a divisor of H): query head h reads kv
    head h // (H // Hkv).  causal: 0 / False, 1 / True (top-left), 2
    (bottom-right); window_left >= 0 adds a sliding window (needs causal)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    _need(cu_seqlens_k, torch.int32, "cu_seqlens_k")
    if (q.dim() != 3 or k.shape != v.shape or k.dim() != 3 or q.shape[2] != k.shape[2] or
            q.shape[1] % k.shape[1] != 0):
        raise ValueError("q, k, v must be [tokens, heads, head_dim]; k/v heads must divide q heads")
    total_q, H, D = q.shape
    Hkv = k.shape[1]
    total_k = k.shape[0]
    batch = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != batch + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((total_q, H), dtype=torch.float32, device=q.device)
    _need(out, torch.bfloat16, "out")
    _need(lse, torch.float32, "lse")
    if workspace is None:
        workspace = alloc_workspace(batch, total_q, total_k, H, D, device=q.device)
    st = lib().vfa_varlen_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                              total_q, total_k, int(max_seqlen_q), batch, H, Hkv, D,
                              float(softmax_scale), int(causal), int(window_left), _ptr(out),
                              _ptr(lse), _ptr(workspace),
                              workspace.numel() * workspace.element_size(),
                              _stream(stream))
    _check(st)
    return out, lse


def varlen_fwd_fp8(q8: torch.Tensor, k8: torch.Tensor, v: torch.Tensor,
                   cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor, max_seqlen_q: int,
                   softmax_scale: float, descale_q: float, descale_k: float, causal,
                   out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None, stream=None,
                   window_left: int = -1):
    """vfa_varlen_fwd_fp8: q8, k8 uint8 E4M3 codes [T, H(kv), 128], v bf16; returns (out, lse)."""
    for t, n in ((q8, "q8"), (k8, "k8")):
        _need(t, torch.uint8, n)
    _need(v, torch.bfloat16, "v")
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    _need(cu_seqlens_k, torch.int32, "cu_seqlens_k")
    if (q8.dim() != 3 or k8.shape != v.shape or q8.shape[2] != k8.shape[2] or
            q8.shape[1] % k8.shape[1] != 0):
        raise ValueError("q8 [Tq, H, D], k8 and v [Tk, Hkv, D] with Hkv dividing H")
    total_q, H, D = q8.shape
    total_k, Hkv = k8.shape[0], k8.shape[1]
    batch = cu_seqlens_q.numel() - 1
    out = torch.empty(q8.shape, dtype=torch.bfloat16, device=q8.device) if out is None else out
    if lse is None:
        lse = torch.empty((total_q, H), dtype=torch.float32, device=q8.device)
    _need(out, torch.bfloat16, "out")
    _need(lse, torch.float32, "lse")
    if workspace is None:
        workspace = alloc_workspace(batch, total_q, total_k, H, D, device=q8.device)
    st = lib().vfa_varlen_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v), _ptr(cu_seqlens_q),
                                  _ptr(cu_seqlens_k), total_q, total_k, int(max_seqlen_q), batch,
                                  H, Hkv, D, float(softmax_scale), float(descale_q),
                                  float(descale_k), int(causal), int(window_left), _ptr(out),
                                  _ptr(lse), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st)
    return out, lse


def alloc_bwd_workspace(batch: int, total_q: int, num_heads: int, head_dim: int,
                        device="cuda") -> torch.Tensor:
    n = lib().vfa_varlen_bwd_workspace_bytes(batch, total_q, num_heads, head_dim)
    if n == 0:
        raise VfaError(VFA_ERR_UNSUPPORTED, "backward workspace size query rejected its arguments")
    return torch.empty(n, dtype=torch.uint8, device=device)


def varlen_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor,
               dout: torch.Tensor, lse: torch.Tensor, cu_seqlens_q: torch.Tensor,
               cu_seqlens_k: torch.Tensor, softmax_scale: float, causal,
               window_left: int = -1, dq: Optional[torch.Tensor] = None,
               dk: Optional[torch.Tensor] = None, dv: Optional[torch.Tensor] = None,
               workspace: Optional[torch.Tensor] = None, stream=None):
    """(dq, dk, dv) bf16 = gradients of varlen_fwd for upstream gradient dout (vfa_varlen_bwd)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse")
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    _need(cu_seqlens_k, torch.int32, "cu_seqlens_k")
    if (q.dim() != 3 or k.shape != v.shape or out.shape != q.shape or dout.shape != q.shape or
            q.shape[2] != k.shape[2] or q.shape[1] % k.shape[1] != 0):
        raise ValueError("q, out, dout [Tq, H, D] and k, v [Tk, Hkv, D] with Hkv dividing H")
    total_q, H, D = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    batch = cu_seqlens_q.numel() - 1
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _need(t, torch.bfloat16, n)
    if workspace is None:
        workspace = alloc_bwd_workspace(batch, total_q, H, D, device=q.device)
    st = lib().vfa_varlen_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                              _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), total_q, total_k, batch, H,
                              Hkv, D, float(softmax_scale), int(causal), int(window_left),
                              _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st)
    return dq, dk, dv, workspace


def varlen_fwd_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                       cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor, max_seqlen_q: int,
                       softmax_scale: float, causal: bool, out: torch.Tensor, lse: torch.Tensor,
                       device_status: Optional[torch.Tensor] = None, stream=None,
                       window_left: int = -1):
    """vfa_varlen_fwd_noalloc: the forward with the library's static scratch.

    For callers that cannot allocate device memory: the caller passes only
    inputs and outputs (allocated however it likes); the library allocates
    nothing.  Calls that can overlap on the GPU must not use it concurrently.
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse")
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    _need(cu_seqlens_k, torch.int32, "cu_seqlens_k")
    total_q, H, D = q.shape
    st = lib().vfa_varlen_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q),
                                      _ptr(cu_seqlens_k), total_q, k.shape[0], int(max_seqlen_q),
                                      cu_seqlens_q.numel() - 1, H, k.shape[1], D,
                                      float(softmax_scale),
                                      int(causal), int(window_left), _ptr(out), _ptr(lse),
                                      _ptr(device_status),
                                      _stream(stream))
    _check(st)
    return out, lse


def schedule(cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor, total_q: int, total_k: int,
             max_seqlen_q: int, num_heads: int, block_q: int, block_k: int, causal: bool,
             pair: bool = False, stream=None, window_left: int = -1):
    """Runs the device tile scheduler alone; returns (items int32 [n, 8] on device, status)."""
    batch = cu_seqlens_q.numel() - 1
    cap = num_heads * (total_q // block_q + batch)
    dev = cu_seqlens_q.device
    items = torch.full((max(cap, 1), 8), -7, dtype=torch.int32, device=dev)
    n_items = torch.zeros(1, dtype=torch.int32, device=dev)
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    # scratch of vfa_varlen_fwd_workspace_bytes() bytes covers any tile shape
    nbytes = workspace_bytes(batch, total_q, total_k, num_heads, 128)
    scratch = torch.empty((nbytes + 3) // 4, dtype=torch.int32, device=dev)
    st = lib().vfa_varlen_schedule(_ptr(cu_seqlens_q), _ptr(cu_seqlens_k), total_q, total_k,
                                   int(max_seqlen_q), batch, num_heads, block_q, block_k,
                                   int(causal), int(window_left), int(bool(pair)), _ptr(items),
                                   cap,
                                   _ptr(n_items), _ptr(status), _ptr(scratch), scratch.numel() * 4,
                                   _stream(stream))
    _check(st)
    n = int(n_items.item())
    return items[:n], int(status.item())


def read_status(word: torch.Tensor, stream=None) -> int:
    """The int32 at word.data_ptr() (workspace status word or decode status)."""
    out = ctypes.c_int32()
    _check(lib().vfa_read_status(_ptr(word), _stream(stream), ctypes.byref(out)))
    return int(out.value)


# ----------------------------------------------------------------- paged decode

def decode_init(m: torch.Tensor, l: torch.Tensor, o: torch.Tensor,
                status: Optional[torch.Tensor] = None, stream=None):
    S, Hq, D = o.shape
    for t, n in ((m, "m"), (l, "l"), (o, "o")):
        _need(t, torch.float32, n)
    _check(lib().vfa_paged_decode_init(_ptr(m), _ptr(l), _ptr(o), S, Hq, D, _ptr(status),
                                       _stream(stream)))


def decode_step(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                tile_blocks: torch.Tensor, tile_block_counts: torch.Tensor,
                m: torch.Tensor, l: torch.Tensor, o: torch.Tensor,
                status: Optional[torch.Tensor] = None, stream=None,
                tile_token_counts: Optional[torch.Tensor] = None, softmax_scale: float = 0.0):
    """vfa_paged_decode_step; tile_token_counts (int32 [S], optional) and
    softmax_scale (<= 0: 1/sqrt(D)) as in include/vfa.h."""
    _need(q, torch.bfloat16, "q")
    if tile_token_counts is not None:
        _need(tile_token_counts, torch.int32, "tile_token_counts")
    _need(k_pool, torch.bfloat16, "k_pool")
    _need(v_pool, torch.bfloat16, "v_pool")
    _need(tile_blocks, torch.int32, "tile_blocks")
    _need(tile_block_counts, torch.int32, "tile_block_counts")
    S, Hq, D = q.shape
    nb, bs, Hkv, D2 = k_pool.shape
    if D2 != D or v_pool.shape != k_pool.shape or tile_blocks.shape[0] != S:
        raise ValueError("inconsistent decode shapes")
    _check(lib().vfa_paged_decode_step(_ptr(q), _ptr(k_pool), _ptr(v_pool), nb, _ptr(tile_blocks),
                                       _ptr(tile_block_counts), _ptr(tile_token_counts),
                                       tile_blocks.shape[1], S, Hq, Hkv, D, bs,
                                       float(softmax_scale), _ptr(m), _ptr(l), _ptr(o),
                                       _ptr(status), _stream(stream)))


def decode_split_count(num_seqs: int, num_kv_heads: int, tile_capacity: int) -> int:
    """vfa_paged_decode_split_count: a run count for the current device."""
    n = ctypes.c_int()
    _check(lib().vfa_paged_decode_split_count(num_seqs, num_kv_heads, tile_capacity,
                                              ctypes.byref(n)))
    return n.value


def alloc_decode_split_workspace(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                 head_dim: int, num_splits: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace for vfa_paged_decode_step_split (the tickets start at zero)."""
    n = lib().vfa_paged_decode_split_workspace_bytes(num_seqs, num_q_heads, num_kv_heads,
                                                     head_dim, num_splits)
    if n == 0:
        raise VfaError(VFA_ERR_UNSUPPORTED, "no split workspace for these sizes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def decode_step_split(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                      tile_blocks: torch.Tensor, tile_block_counts: torch.Tensor,
                      m: torch.Tensor, l: torch.Tensor, o: torch.Tensor, num_splits: int,
                      workspace: torch.Tensor, status: Optional[torch.Tensor] = None,
                      stream=None, tile_token_counts: Optional[torch.Tensor] = None,
                      softmax_scale: float = 0.0):
    """vfa_paged_decode_step_split: the step with each tile cut into num_splits runs."""
    _need(q, torch.bfloat16, "q")
    if tile_token_counts is not None:
        _need(tile_token_counts, torch.int32, "tile_token_counts")
    _need(k_pool, torch.bfloat16, "k_pool")
    _need(v_pool, torch.bfloat16, "v_pool")
    _need(tile_blocks, torch.int32, "tile_blocks")
    _need(tile_block_counts, torch.int32, "tile_block_counts")
    _need(workspace, torch.uint8, "workspace")
    S, Hq, D = q.shape
    nb, bs, Hkv, D2 = k_pool.shape
    if D2 != D or v_pool.shape != k_pool.shape or tile_blocks.shape[0] != S:
        raise ValueError("inconsistent decode shapes")
    _check(lib().vfa_paged_decode_step_split(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), nb, _ptr(tile_blocks), _ptr(tile_block_counts),
        _ptr(tile_token_counts), tile_blocks.shape[1], S, Hq, Hkv, D, bs, float(softmax_scale),
        _ptr(m), _ptr(l), _ptr(o), _ptr(status), int(num_splits), _ptr(workspace),
        workspace.numel(), _stream(stream)))


def decode_finalize(l: torch.Tensor, o: torch.Tensor, out: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    S, Hq, D = o.shape
    if out is None:
        out = torch.empty((S, Hq, D), dtype=torch.bfloat16, device=o.device)
    _check(lib().vfa_paged_decode_finalize(_ptr(l), _ptr(o), S, Hq, D, _ptr(out),
                                           _stream(stream)))
    return out


def debug_bounded_wait(status: torch.Tensor, stream=None):
    """vfa_debug_bounded_wait: a wait nothing satisfies must end in VFA_ERR_TIMEOUT."""
    _need(status, torch.int32, "status")
    _check(lib().vfa_debug_bounded_wait(_ptr(status), _stream(stream)))


def debug_paged_gather(k_pool: torch.Tensor, v_pool: torch.Tensor, tile_blocks: torch.Tensor,
                       tile_block_counts: torch.Tensor, k_out: torch.Tensor, v_out: torch.Tensor,
                       status: Optional[torch.Tensor] = None, stream=None):
    nb, bs, Hkv, D = k_pool.shape
    S, cap = tile_blocks.shape
    _check(lib().vfa_debug_paged_gather(_ptr(k_pool), _ptr(v_pool), nb, _ptr(tile_blocks),
                                        _ptr(tile_block_counts), cap, S, Hkv, D, bs,
                                        _ptr(k_out), _ptr(v_out), _ptr(status), _stream(stream)))
