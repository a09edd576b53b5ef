"""fp64 CPU oracle for the H3 attention hot path.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by ``bench.py``'s CPU-baseline / reference leg.  The product package never
imports it, and it never imports the product package.

The arithmetic lives in ``h3_oracle.c`` (plain C, fp64, OpenMP); this module
only marshals numpy arrays into it.  Each function names the passage it
follows in the C source's header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "h3_oracle.c")
_LIB = os.path.join(_HERE, "libh3oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, no FMA contraction, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        d, i64, i32 = ctypes.c_double, ctypes.c_int64, ctypes.c_int
        p = ctypes.c_void_p
        lib.h3o_rmsnorm.argtypes = [p, p, i64, i32, d, p]
        lib.h3o_rope.argtypes = [p, p, i64, i32, i32, i32, i32, i32, d, i32, p]
        lib.h3o_attention.argtypes = [p, i64, p, p, i64, i32, i32, i64, d, p]
        lib.h3o_seq2head_u16.argtypes = [p, p, i64, i32, i32, i32]
        lib.h3o_head2seq_u16.argtypes = [p, p, i64, i32, i32, i32]
        lib.h3o_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.h3o_e4m3_decode.restype = d
        lib.h3o_qkv_proj_fp8.argtypes = [p, i64, p, i32, i32, i32, i32, d, p]
        lib.h3o_qkv_proj_fp8.restype = None
        lib.h3o_num_threads.restype = i32
        for f in (lib.h3o_rmsnorm, lib.h3o_rope, lib.h3o_attention,
                  lib.h3o_seq2head_u16, lib.h3o_head2seq_u16):
            f.restype = None
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().h3o_num_threads())


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def rmsnorm(x, w, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * w."""
    x = _f64(x)
    w = _f64(w)
    D = x.shape[-1]
    assert w.shape == (D,)
    y = np.empty_like(x)
    _load().h3o_rmsnorm(_ptr(x), _ptr(w), x.size // D, D, float(eps), _ptr(y))
    return y


def rope(x, pos, d_t: int, d_h: int, d_w: int, theta: float = 10000.0,
         interleaved: bool = True) -> np.ndarray:
    """Three-axis rotary embedding of x [S, H, D] by pos int32 [S, 3]."""
    x = _f64(x)
    S, H, D = x.shape
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    assert pos.shape == (S, 3)
    assert d_t % 2 == 0 and d_h % 2 == 0 and d_w % 2 == 0 and d_t + d_h + d_w <= D
    y = np.empty_like(x)
    _load().h3o_rope(_ptr(x), _ptr(pos), S, H, D, d_t, d_h, d_w, float(theta),
                     1 if interleaved else 0, _ptr(y))
    return y


def attention(q, k, v, kv_len: int | None = None, scale: float | None = None) -> np.ndarray:
    """Exact softmax attention per head over keys [0, kv_len).

    q [Sq, H, D] (any subset of query rows), k and v [S, H, D] -> o [Sq, H, D].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    Sq, H, D = q.shape
    S = k.shape[0]
    assert k.shape == (S, H, D) and v.shape == (S, H, D)
    kv = S if kv_len is None else int(kv_len)
    assert 1 <= kv <= S
    sc = 1.0 / np.sqrt(D) if scale is None else float(scale)
    o = np.empty((Sq, H, D), dtype=np.float64)
    _load().h3o_attention(_ptr(q), Sq, _ptr(k), _ptr(v), S, H, D, kv, sc, _ptr(o))
    return o


def seq2head(x_u16, P: int) -> np.ndarray:
    """[S, H, D] 16-bit words (P sequence shards) -> [P, S, H/P, D]."""
    x = np.ascontiguousarray(x_u16, dtype=np.uint16)
    S, H, D = x.shape
    assert S % P == 0 and H % P == 0
    out = np.empty((P, S, H // P, D), dtype=np.uint16)
    _load().h3o_seq2head_u16(_ptr(x), _ptr(out), S, H, D, P)
    return out


def head2seq(x_u16, P: int) -> np.ndarray:
    """[P, S, H/P, D] 16-bit words -> [S, H, D] (P sequence shards)."""
    x = np.ascontiguousarray(x_u16, dtype=np.uint16)
    P_, S, Hp, D = x.shape
    assert P_ == P and S % P == 0
    out = np.empty((S, Hp * P, D), dtype=np.uint16)
    _load().h3o_head2seq_u16(_ptr(x), _ptr(out), S, Hp * P, D, P)
    return out


def e4m3_decode(code: int) -> float:
    """Value of one FP8 E4M3 code (NaN for S.1111.111)."""
    return float(_load().h3o_e4m3_decode(int(code) & 0xFF))


def qkv_proj_fp8(x_codes, w_codes, scale: float, inner: int, P: int, rank: int) -> np.ndarray:
    """Projection of the given rows of x ([n, hidden] E4M3 codes) through rank
    `rank`'s head rows of w ([3*inner, hidden] E4M3 codes), times `scale`.
    Returns [n, 3, inner/P] float64 (q, k, v parts)."""
    x = np.ascontiguousarray(x_codes, dtype=np.uint8)
    w = np.ascontiguousarray(w_codes, dtype=np.uint8)
    n, hidden = x.shape
    assert w.shape == (3 * inner, hidden) and inner % P == 0 and 0 <= rank < P
    out = np.empty((n, 3, inner // P), dtype=np.float64)
    _load().h3o_qkv_proj_fp8(_ptr(x), n, _ptr(w), hidden, inner, P, rank, float(scale), _ptr(out))
    return out


def norm_rope(x, w, pos, eps: float, d_t: int, d_h: int, d_w: int,
              theta: float = 10000.0, interleaved: bool = True) -> np.ndarray:
    """QK-norm after the head split, then the rotary embedding ([S, H, D])."""
    return rope(rmsnorm(x, w, eps), pos, d_t, d_h, d_w, theta, interleaved)


def bf16_to_f64(t) -> np.ndarray:
    """Exact widening of a bf16 torch tensor (any device) to a float64 array."""
    import torch
    return t.detach().to("cpu").to(torch.float64).numpy()


def bf16_bits(t) -> np.ndarray:
    """The raw 16-bit words of a bf16 torch tensor, as uint16."""
    import torch
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
