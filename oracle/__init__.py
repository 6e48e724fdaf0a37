"""Oracle -- TEST INFRASTRUCTURE ONLY.

A plain, slow CPU statement (fp64 for floating point, plain integers for the
tile schedule) of what the variable-length attention path computes.  Only the
test-suite, the package's ``smoke()`` check and the bench's CPU-baseline leg
may import this package.  The product path (the CUDA library and its Python
binding) never imports, links or executes anything here, and this package
shares no code with it.

Pages followed:
  * "Varlen Flash Attention Implementation Plan" (rustytorch): Task 1 Step 1
    (the kernel's layout, masks and epilogue) and Task 2 Step 1
    (``varlen_attention_cpu``).
  * "attention_ref.rs" (spark_storage): ``AttnState::new``,
    ``step_tile_ref`` and ``finalize_ref``.

Where the pages only name a variant, the oracle states the plainest reading:
the backward is the exact derivative of the forward (``varlen_bwd``); the FP8
forward reads E4M3 codes as descale * code exactly (``varlen_fwd_fp8``); the
sliding window hides keys below row + off - window_left.

``vfa_oracle.c`` holds the floating-point definitions; ``schedule.py`` holds
the integer tile-schedule rule.  Parity pins for every function are in
``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vfa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libvfa_oracle.so")
_lock = threading.Lock()
_lib = None

FLT_MAX = float(np.finfo(np.float32).max)


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_default_threads.restype = i32
        lib.oracle_varlen_fwd.argtypes = [P, P, P, P, P, i32, i32, i32, i32, f64, i32, i32, P, P,
                                          i32]
        lib.oracle_varlen_fwd.restype = i32
        lib.oracle_varlen_fwd_rows.argtypes = [P, P, P, P, P, i32, i32, i32, i32, f64, i32, i32,
                                               P, i64, P, P, i32]
        lib.oracle_varlen_fwd_rows.restype = i32
        lib.oracle_varlen_bwd.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, f64, i32, i32, P,
                                          P, P, i32]
        lib.oracle_varlen_bwd.restype = i32
        lib.oracle_varlen_fwd_fp8.argtypes = [P, P, P, P, P, i32, i32, i32, i32, f64, f64, f64,
                                              i32, i32, P, P, i32]
        lib.oracle_varlen_fwd_fp8.restype = i32
        lib.oracle_fp8_e4m3_decode.argtypes = [P, i64, P]
        lib.oracle_fp8_e4m3_decode.restype = None
        lib.oracle_decode_init.argtypes = [P, P, P, i32, i32, i32]
        lib.oracle_decode_init.restype = None
        lib.oracle_decode_step.argtypes = [P, P, P, i64, P, P, P, i32, i32, i32, i32, i32, i32,
                                           f64, P, P, P, i32]
        lib.oracle_decode_step.restype = i32
        lib.oracle_decode_finalize.argtypes = [P, P, i32, i32, i32, P]
        lib.oracle_decode_finalize.restype = None
        _lib = lib
        return lib


def _bits(x) -> np.ndarray:
    """bf16 values (a torch bfloat16 tensor, or uint16 bit patterns) -> contiguous uint16."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy inputs must be uint16 bfloat16 bit patterns")
        return np.ascontiguousarray(x)
    import torch
    if x.dtype != torch.bfloat16:
        raise TypeError("expected a bfloat16 tensor")
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy()).view(np.uint16)


def _i32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def varlen_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, num_heads: int, head_dim: int,
               softmax_scale: float, causal: bool, nthreads: int = 0,
               num_kv_heads: int = 0, window_left: int = -1):
    """Full forward.  Returns (out float64 [Tq,H,D], lse float64 [Tq,H], threads used).

    causal: 0 (or False) no mask, 1 (or True) top-left, 2 bottom-right (local
    key j visible to local query i iff j <= i + Lk - Lq); window_left >= 0
    (with a causal mode) also hides keys j < i + off - window_left.  k, v hold
    num_kv_heads heads (default: num_heads); query head h reads kv head
    h // (num_heads // num_kv_heads)."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    cq, ck = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    batch = len(cq) - 1
    tq = int(cq[-1])
    hkv = num_kv_heads or num_heads
    if qb.size != tq * num_heads * head_dim:
        raise ValueError("q size does not match cu_seqlens_q[-1] * H * D")
    if kb.size != int(ck[-1]) * hkv * head_dim or vb.size != kb.size:
        raise ValueError("k/v size does not match cu_seqlens_k[-1] * Hkv * D")
    out = np.zeros((tq, num_heads, head_dim), dtype=np.float64)
    lse = np.zeros((tq, num_heads), dtype=np.float64)
    n = lib.oracle_varlen_fwd(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(cq), _ptr(ck), batch,
                              num_heads, hkv, head_dim, float(softmax_scale),
                              int(causal), int(window_left), _ptr(out), _ptr(lse), int(nthreads))
    if n <= 0:
        raise ValueError(f"oracle_varlen_fwd rejected its arguments ({n})")
    return out, lse, int(n)


def varlen_fwd_rows(q, k, v, cu_seqlens_q, cu_seqlens_k, num_heads: int, head_dim: int,
                    softmax_scale: float, causal: bool, rows, nthreads: int = 0,
                    num_kv_heads: int = 0, window_left: int = -1):
    """Selected rows.  rows: int array [n, 2] of (packed token, head).

    Returns (out float64 [n, D], lse float64 [n], threads used)."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    cq, ck = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
    out = np.zeros((r.shape[0], head_dim), dtype=np.float64)
    lse = np.zeros((r.shape[0],), dtype=np.float64)
    n = lib.oracle_varlen_fwd_rows(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(cq), _ptr(ck),
                                   len(cq) - 1, num_heads, num_kv_heads or num_heads, head_dim,
                                   float(softmax_scale),
                                   int(causal), int(window_left), _ptr(r), r.shape[0], _ptr(out),
                                   _ptr(lse),
                                   int(nthreads))
    if n <= 0:
        raise ValueError(f"oracle_varlen_fwd_rows rejected its arguments ({n})")
    return out, lse, int(n)


def _u8(a) -> np.ndarray:
    if isinstance(a, np.ndarray):
        return np.ascontiguousarray(a.view(np.uint8))
    import torch
    return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.uint8).numpy())


def fp8_e4m3_decode(codes) -> np.ndarray:
    """Exact float64 values of FP8 E4M3 codes (uint8 array or a float8_e4m3fn tensor)."""
    c = _u8(codes)
    out = np.zeros(c.shape, dtype=np.float64)
    _load().oracle_fp8_e4m3_decode(_ptr(c), c.size, _ptr(out))
    return out


def varlen_fwd_fp8(q8, k8, v, cu_seqlens_q, cu_seqlens_k, num_heads: int, head_dim: int,
                   softmax_scale: float, descale_q: float, descale_k: float, causal,
                   nthreads: int = 0, num_kv_heads: int = 0, window_left: int = -1):
    """Forward with FP8 E4M3 q and k (codes, one descale per tensor) and bf16 v.

    Returns (out float64 [Tq,H,D], lse float64 [Tq,H], threads used)."""
    lib = _load()
    qb, kb, vb = _u8(q8), _u8(k8), _bits(v)
    cq, ck = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    batch = len(cq) - 1
    tq = int(cq[-1])
    hkv = num_kv_heads or num_heads
    if qb.size != tq * num_heads * head_dim:
        raise ValueError("q size does not match cu_seqlens_q[-1] * H * D")
    if kb.size != int(ck[-1]) * hkv * head_dim or vb.size != kb.size:
        raise ValueError("k/v size does not match cu_seqlens_k[-1] * Hkv * D")
    out = np.zeros((tq, num_heads, head_dim), dtype=np.float64)
    lse = np.zeros((tq, num_heads), dtype=np.float64)
    n = lib.oracle_varlen_fwd_fp8(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(cq), _ptr(ck), batch,
                                  num_heads, hkv, head_dim, float(softmax_scale),
                                  float(descale_q), float(descale_k), int(causal),
                                  int(window_left), _ptr(out), _ptr(lse), int(nthreads))
    if n <= 0:
        raise ValueError(f"oracle_varlen_fwd_fp8 rejected its arguments ({n})")
    return out, lse, int(n)


def varlen_bwd(q, k, v, dout, cu_seqlens_q, cu_seqlens_k, num_heads: int, head_dim: int,
               softmax_scale: float, causal, nthreads: int = 0, num_kv_heads: int = 0,
               window_left: int = -1):
    """Gradients of the forward for upstream gradient dout.

    Returns (dq float64 [Tq,H,D], dk float64 [Tk,Hkv,D], dv float64 [Tk,Hkv,D],
    threads used); masks and head grouping as in varlen_fwd."""
    lib = _load()
    qb, kb, vb, gb = _bits(q), _bits(k), _bits(v), _bits(dout)
    cq, ck = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    batch = len(cq) - 1
    tq, tk = int(cq[-1]), int(ck[-1])
    hkv = num_kv_heads or num_heads
    if qb.size != tq * num_heads * head_dim or gb.size != qb.size:
        raise ValueError("q / dout size does not match cu_seqlens_q[-1] * H * D")
    if kb.size != tk * hkv * head_dim or vb.size != kb.size:
        raise ValueError("k/v size does not match cu_seqlens_k[-1] * Hkv * D")
    dq = np.zeros((tq, num_heads, head_dim), dtype=np.float64)
    dk = np.zeros((tk, hkv, head_dim), dtype=np.float64)
    dv = np.zeros((tk, hkv, head_dim), dtype=np.float64)
    n = lib.oracle_varlen_bwd(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(gb), _ptr(cq), _ptr(ck), batch,
                              num_heads, hkv, head_dim, float(softmax_scale), int(causal),
                              int(window_left), _ptr(dq), _ptr(dk), _ptr(dv), int(nthreads))
    if n <= 0:
        raise ValueError(f"oracle_varlen_bwd rejected its arguments ({n})")
    return dq, dk, dv, int(n)


class DecodeState:
    """fp64 (m, l, o) -- AttnState of attention_ref.rs, kept in double."""

    def __init__(self, num_seqs: int, num_q_heads: int, head_dim: int):
        self.num_seqs, self.num_q_heads, self.head_dim = num_seqs, num_q_heads, head_dim
        self.m = np.empty((num_seqs, num_q_heads), dtype=np.float64)
        self.l = np.empty((num_seqs, num_q_heads), dtype=np.float64)
        self.o = np.empty((num_seqs, num_q_heads, head_dim), dtype=np.float64)
        _load().oracle_decode_init(_ptr(self.m), _ptr(self.l), _ptr(self.o),
                                   num_seqs, num_q_heads, head_dim)

    def copy(self) -> "DecodeState":
        c = DecodeState.__new__(DecodeState)
        c.num_seqs, c.num_q_heads, c.head_dim = self.num_seqs, self.num_q_heads, self.head_dim
        c.m, c.l, c.o = self.m.copy(), self.l.copy(), self.o.copy()
        return c


def decode_step(state: DecodeState, q, k_pool, v_pool, tile_blocks, tile_block_counts,
                num_kv_heads: int, block_size: int, nthreads: int = 0,
                tile_token_counts=None, scale: float = 0.0) -> int:
    """One step_tile over every sequence; updates `state` in place.  Returns threads used.

    tile_token_counts (optional, [S]): absorb only the first n tokens of each
    sequence's listed blocks; scale <= 0 means 1/sqrt(head_dim)."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k_pool), _bits(v_pool)
    tb = _i32(tile_blocks)
    tc = _i32(tile_block_counts)
    tt = None if tile_token_counts is None else _i32(tile_token_counts)
    S, Hq, D = state.num_seqs, state.num_q_heads, state.head_dim
    cap = tb.shape[1] if tb.ndim == 2 else (tb.size // S if S else 0)
    per_block = block_size * num_kv_heads * D
    num_blocks = kb.size // per_block
    if kb.size != num_blocks * per_block or vb.size != kb.size or qb.size != S * Hq * D:
        raise ValueError("decode_step: inconsistent buffer sizes")
    n = lib.oracle_decode_step(_ptr(qb), _ptr(kb), _ptr(vb), num_blocks, _ptr(tb), _ptr(tc),
                               None if tt is None else _ptr(tt), int(cap), S, Hq, num_kv_heads,
                               D, block_size, float(scale), _ptr(state.m), _ptr(state.l),
                               _ptr(state.o), int(nthreads))
    if n <= 0:
        raise ValueError(f"oracle_decode_step rejected its arguments ({n})")
    return int(n)


def decode_finalize(state: DecodeState) -> np.ndarray:
    """finalize_ref in double: out = o / l (0 where l = 0).  Returns float64 [S, Hq, D]."""
    out = np.empty_like(state.o)
    _load().oracle_decode_finalize(_ptr(state.l), _ptr(state.o), state.num_seqs,
                                   state.num_q_heads, state.head_dim, _ptr(out))
    return out


from .schedule import schedule, tile_cost  # noqa: E402  (integer rule, pure Python)

__all__ = ["build", "default_threads", "varlen_fwd", "varlen_fwd_rows", "varlen_bwd",
           "varlen_fwd_fp8", "fp8_e4m3_decode", "DecodeState",
           "decode_step", "decode_finalize", "schedule", "tile_cost", "FLT_MAX"]
