"""GB300 (sm_103a) attention hot path of a MiniMax-H3-style DiT block.

Thin Python binding over ``libh3attn.so`` (C ABI in ``include/h3attn.h``).
The functions here only check and marshal torch tensors into the C calls of
the same names; every step of the path runs in the library's CUDA kernels.
There is no fallback: if the library is missing or the device is not an
sm_103 GPU, calls raise.

Two builds of the same kernels exist: ``libh3attn.so`` and
``libh3attn_debug.so``, in which every kernel checks its computed indices and
reports a failed check as H3ATTN_ERR_DEVICE_BOUNDS instead of touching memory
outside its buffers.  The debug build is used when the environment variable
``H3ATTN_DEBUG`` is ``1`` at the first call, or after ``use_debug_checks(True)``.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "H3AttnError", "load_library", "library_path",
    "h3attn_qk_norm_rope", "h3attn_qk_norm_rope_seq2head", "h3attn_forward", "h3attn_seq2head",
    "h3attn_head2seq", "h3attn_head2seq_heads", "h3attn_qkv_proj_fp8",
    "h3attn_get_device_status", "h3attn_strerror", "h3attn_version", "h3attn_selftest_wait_timeout",
    "h3attn_last_device_error_info", "h3attn_build_flags", "h3attn_selftest_bounds", "use_debug_checks",
    "ulysses_attention_step", "make_workspace", "StepGraph",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATHS = {False: os.path.join(_PKG, "libh3attn.so"), True: os.path.join(_PKG, "libh3attn_debug.so")}
_libs = {}
_debug = os.environ.get("H3ATTN_DEBUG", "") == "1"

H3ATTN_OK = 0
H3ATTN_ERR_ARG = -1
H3ATTN_ERR_SHAPE = -2
H3ATTN_ERR_ALIAS = -3
H3ATTN_ERR_CUDA = -4
H3ATTN_ERR_DEVICE_TIMEOUT = -5
H3ATTN_ERR_UNSUPPORTED_DEVICE = -6
H3ATTN_ERR_DEVICE_BOUNDS = -7
H3ATTN_BUILD_DEBUG_CHECKS = 1

# exported symbol -> (restype, argtypes)
_P, _I, _F, _U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_ulonglong
SIGNATURES = {
    "h3attn_qk_norm_rope": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _F, _P]),
    "h3attn_forward": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _F, _P]),
    "h3attn_qk_norm_rope_seq2head": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _F, _P]),
    "h3attn_head2seq_heads": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _P]),
    "h3attn_qkv_proj_fp8": (_I, [_P, _P, _F, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "h3attn_seq2head": (_I, [_P, _P, _I, _I, _I, _I, _P]),
    "h3attn_head2seq": (_I, [_P, _P, _I, _I, _I, _I, _P]),
    "h3attn_get_device_status": (_I, [_P]),
    "h3attn_last_device_error_info": (_U64, []),
    "h3attn_last_cuda_error": (_I, []),
    "h3attn_strerror": (ctypes.c_char_p, [_I]),
    "h3attn_version": (_I, []),
    "h3attn_selftest_wait_timeout": (_I, [_U64, _P]),
    "h3attn_build_flags": (_I, []),
    "h3attn_selftest_bounds": (_I, [_P, _U64, _P]),
}


class H3AttnError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = f"{fn} failed: {code} ({h3attn_strerror(code)})"
        if code == H3ATTN_ERR_CUDA:
            msg += f"; cudaError {load_library().h3attn_last_cuda_error()}"
        super().__init__(msg)
        self.code = code


def library_path() -> str:
    return _LIB_PATHS[_debug]


def use_debug_checks(enable: bool) -> None:
    """Route every following call to libh3attn_debug.so (True) or libh3attn.so
    (False).  Each library keeps its own device status word."""
    global _debug
    _debug = bool(enable)


def load_library():
    """Load the selected build (built in-tree by ``dit_sequence_attention_gb300.build``)."""
    lib = _libs.get(_debug)
    if lib is None:
        path = _LIB_PATHS[_debug]
        if not os.path.exists(path):
            flag = " --debug" if _debug else ""
            raise RuntimeError(f"{path} is not built; run `python -m dit_sequence_attention_gb300.build{flag}` "
                               "(or __graft_entry__.build()) first")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _libs[_debug] = lib
    return lib


def _stream_ptr(stream, device=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


def _on(t: torch.Tensor):
    """Make the tensors' GPU the current device for the call: the library
    launches on the current device and refuses memory of any other."""
    return torch.cuda.device(t.device)


def _check(fn: str, rc: int):
    if rc != H3ATTN_OK:
        raise H3AttnError(fn, rc)


def _bf16(t: torch.Tensor, name: str, device=None):
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _bshd(t: torch.Tensor, name: str):
    if t.dim() == 3:
        return (1, *t.shape)
    if t.dim() == 4:
        return tuple(t.shape)
    raise ValueError(f"{name} must be [S, H, D] or [B, S, H, D]")


def h3attn_strerror(code: int) -> str:
    return load_library().h3attn_strerror(int(code)).decode()


def h3attn_version() -> int:
    return int(load_library().h3attn_version())


def h3attn_qk_norm_rope(q, k, q_out, k_out, w_q, w_k, pos, d_t, d_h, d_w, eps=1e-6, theta=10000.0,
                        dbg_fp32=None, stream=None):
    """QK-RMSNorm then 3-axis RoPE of q and k ([S,H,D] or [B,S,H,D] bf16); in place if q_out is q."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (q_out, "q_out"), (k_out, "k_out")):
        _bf16(t, n, q.device)
    B, S, H, D = _bshd(q, "q")
    for t, n in ((k, "k"), (q_out, "q_out"), (k_out, "k_out")):
        if _bshd(t, n) != (B, S, H, D):
            raise ValueError(f"{n} shape {tuple(t.shape)} != q shape {tuple(q.shape)}")
    for t, n in ((w_q, "w_q"), (w_k, "w_k")):
        if t.dtype != torch.float32 or t.device != q.device or t.numel() != D or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous fp32 [D] tensor on {q.device}")
    if pos.dtype != torch.int32 or pos.device != q.device or tuple(pos.shape) != (S, 3) or not pos.is_contiguous():
        raise ValueError(f"pos must be a contiguous int32 [S, 3] tensor on {q.device}")
    dbg = None
    if dbg_fp32 is not None:
        if dbg_fp32.dtype != torch.float32 or dbg_fp32.numel() != 2 * B * S * H * D or not dbg_fp32.is_contiguous():
            raise ValueError("dbg_fp32 must be a contiguous fp32 tensor of 2*B*S*H*D elements")
        dbg = dbg_fp32.data_ptr()
    with _on(q):
        rc = lib.h3attn_qk_norm_rope(q.data_ptr(), k.data_ptr(), q_out.data_ptr(), k_out.data_ptr(), dbg,
                                     w_q.data_ptr(), w_k.data_ptr(), pos.data_ptr(), B, S, H, D, d_t, d_h, d_w,
                                     float(eps), float(theta), _stream_ptr(stream, q.device))
    _check("h3attn_qk_norm_rope", rc)


def h3attn_qk_norm_rope_seq2head(q, k, qh_out, kh_out, w_q, w_k, pos, P, d_t, d_h, d_w, eps=1e-6,
                                 theta=10000.0, dbg_fp32=None, stream=None):
    """QK-norm + RoPE of [S,H,D] q and k written straight into the head-sharded [P,S,H/P,D] layout."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (qh_out, "qh_out"), (kh_out, "kh_out")):
        _bf16(t, n, q.device)
    if q.dim() != 3 or k.shape != q.shape:
        raise ValueError("q and k must be [S, H, D] of the same shape")
    S, H, D = q.shape
    if H % P or S % P:
        raise ValueError(f"P={P} must divide S={S} and H={H}")
    for t, n in ((qh_out, "qh_out"), (kh_out, "kh_out")):
        if tuple(t.shape) != (P, S, H // P, D):
            raise ValueError(f"{n} must be [P, S, H/P, D] = {(P, S, H // P, D)}")
    for t, n in ((w_q, "w_q"), (w_k, "w_k")):
        if t.dtype != torch.float32 or t.device != q.device or t.numel() != D or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous fp32 [D] tensor on {q.device}")
    if pos.dtype != torch.int32 or pos.device != q.device or tuple(pos.shape) != (S, 3) or not pos.is_contiguous():
        raise ValueError(f"pos must be a contiguous int32 [S, 3] tensor on {q.device}")
    dbg = None
    if dbg_fp32 is not None:
        if dbg_fp32.dtype != torch.float32 or dbg_fp32.numel() != 2 * S * H * D or not dbg_fp32.is_contiguous():
            raise ValueError("dbg_fp32 must be a contiguous fp32 tensor of 2*S*H*D elements")
        dbg = dbg_fp32.data_ptr()
    with _on(q):
        rc = lib.h3attn_qk_norm_rope_seq2head(q.data_ptr(), k.data_ptr(), qh_out.data_ptr(), kh_out.data_ptr(), dbg,
                                              w_q.data_ptr(), w_k.data_ptr(), pos.data_ptr(), S, H, D, int(P), d_t,
                                              d_h, d_w, float(eps), float(theta), _stream_ptr(stream, q.device))
    _check("h3attn_qk_norm_rope_seq2head", rc)


def h3attn_forward(q, k, v, o, head_begin=0, head_count=None, kv_len=None, scale=0.0, stream=None):
    """Masked softmax attention for heads [head_begin, head_begin + head_count) of [B,]S,H_buf,D tensors.

    kv_len: None (all S), an int (every batch item) or a sequence of B ints.
    """
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o")):
        _bf16(t, n, q.device)
    B, S, H, D = _bshd(q, "q")
    for t, n in ((k, "k"), (v, "v"), (o, "o")):
        if _bshd(t, n) != (B, S, H, D):
            raise ValueError(f"{n} shape {tuple(t.shape)} != q shape {tuple(q.shape)}")
    if head_count is None:
        head_count = H - head_begin
    kv_arr = None
    if kv_len is not None:
        vals = [int(kv_len)] * B if isinstance(kv_len, int) else [int(x) for x in kv_len]
        if len(vals) != B:
            raise ValueError(f"kv_len has {len(vals)} entries, expected {B}")
        kv_arr = (ctypes.c_int32 * B)(*vals)
    with _on(q):
        rc = lib.h3attn_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, S, H, D,
                                int(head_begin), int(head_count),
                                ctypes.cast(kv_arr, ctypes.c_void_p) if kv_arr is not None else None,
                                float(scale), _stream_ptr(stream, q.device))
    _check("h3attn_forward", rc)


def _layout(fn_name, src, dst, S, H, D, P, stream):
    lib = load_library()
    _bf16(src, "in")
    _bf16(dst, "out", src.device)
    if src.numel() != S * H * D or dst.numel() != S * H * D:
        raise ValueError("in/out must hold S*H*D elements")
    with _on(src):
        rc = getattr(lib, fn_name)(src.data_ptr(), dst.data_ptr(), S, H, D, int(P), _stream_ptr(stream, src.device))
    _check(fn_name, rc)


def h3attn_seq2head(x, out, P, stream=None):
    """[S, H, D] (P sequence shards) -> out [P, S, H/P, D]."""
    if x.dim() != 3:
        raise ValueError("x must be [S, H, D]")
    S, H, D = x.shape
    _layout("h3attn_seq2head", x, out, S, H, D, P, stream)


def h3attn_head2seq(x, out, P, stream=None):
    """[P, S, H/P, D] -> out [S, H, D] (P sequence shards)."""
    if x.dim() != 4 or x.shape[0] != P:
        raise ValueError("x must be [P, S, H/P, D]")
    _, S, Hp, D = x.shape
    _layout("h3attn_head2seq", x, out, S, Hp * P, D, P, stream)


def h3attn_head2seq_heads(x_group, out, P, group, head_begin, head_count, stream=None):
    """Heads [head_begin, head_begin+head_count) of group `group` ([S, H/P, D]) -> out [S, H, D]."""
    lib = load_library()
    _bf16(x_group, "in_group")
    _bf16(out, "out", x_group.device)
    if x_group.dim() != 3 or out.dim() != 3:
        raise ValueError("in_group must be [S, H/P, D] and out [S, H, D]")
    S, Hp, D = x_group.shape
    if tuple(out.shape) != (S, Hp * P, D):
        raise ValueError("out must be [S, H, D] with H = P * (H/P)")
    with _on(x_group):
        rc = lib.h3attn_head2seq_heads(x_group.data_ptr(), out.data_ptr(), S, Hp * P, D, int(P), int(group),
                                       int(head_begin), int(head_count), _stream_ptr(stream, x_group.device))
    _check("h3attn_head2seq_heads", rc)


def h3attn_qkv_proj_fp8(x_fp8, w_fp8, scale, q_out, k_out, v_out, P, rank, stream=None):
    """This rank's q, k, v ([S, inner/P] bf16 each) = scale * x_fp8 [S, hidden] @ its head rows of w_fp8.

    x_fp8 / w_fp8: uint8 tensors of FP8 E4M3 codes (or torch.float8_e4m3fn), w_fp8 [3*inner, hidden].
    """
    lib = load_library()
    for t, n in ((x_fp8, "x_fp8"), (w_fp8, "w_fp8")):
        if t.dtype not in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)) or not t.is_cuda \
                or not t.is_contiguous() or t.dim() != 2:
            raise ValueError(f"{n} must be a contiguous 2-D CUDA tensor of E4M3 codes")
    S, hidden = x_fp8.shape
    if w_fp8.shape[1] != hidden or w_fp8.shape[0] % 3:
        raise ValueError("w_fp8 must be [3*inner, hidden]")
    inner = w_fp8.shape[0] // 3
    for t, n in ((q_out, "q_out"), (k_out, "k_out"), (v_out, "v_out")):
        _bf16(t, n, x_fp8.device)
        if t.numel() != S * (inner // P):
            raise ValueError(f"{n} must hold S * inner/P = {S * (inner // P)} elements")
    with _on(x_fp8):
        rc = lib.h3attn_qkv_proj_fp8(x_fp8.data_ptr(), w_fp8.data_ptr(), float(scale), q_out.data_ptr(),
                                     k_out.data_ptr(), v_out.data_ptr(), S, hidden, inner, int(P), int(rank),
                                     _stream_ptr(stream, x_fp8.device))
    _check("h3attn_qkv_proj_fp8", rc)


def h3attn_get_device_status(stream=None) -> int:
    """Take the current device's status word (read and clear it in one atomic
    exchange, ordered after the work already on `stream`), synchronise
    `stream`, and return the status code (0 = ok).  An error recorded by a
    kernel on another stream is returned by this call or by the next one."""
    return int(load_library().h3attn_get_device_status(_stream_ptr(stream)))


def h3attn_last_device_error_info() -> int:
    """Diagnostic word of the last device error taken on the current device
    (kernel tag << 32 | site << 16 | low index bits), 0 if none."""
    return int(load_library().h3attn_last_device_error_info())


def h3attn_selftest_wait_timeout(limit_ns: int, stream=None):
    rc = load_library().h3attn_selftest_wait_timeout(int(limit_ns), _stream_ptr(stream))
    _check("h3attn_selftest_wait_timeout", rc)


def h3attn_build_flags() -> int:
    return int(load_library().h3attn_build_flags())


def h3attn_selftest_bounds(buf: torch.Tensor, stream=None):
    """Self-test of the device index checks (debug build only): ``buf`` is a
    CUDA tensor of at least 1024 bytes, overwritten.  Read the outcome with
    ``h3attn_get_device_status()`` (H3ATTN_ERR_DEVICE_BOUNDS expected)."""
    if not isinstance(buf, torch.Tensor) or not buf.is_cuda or not buf.is_contiguous():
        raise ValueError("buf must be a contiguous CUDA tensor")
    with _on(buf):
        rc = load_library().h3attn_selftest_bounds(buf.data_ptr(), buf.numel() * buf.element_size(),
                                                   _stream_ptr(stream, buf.device))
    _check("h3attn_selftest_bounds", rc)


def ulysses_attention_step(q, k, v, w_q, w_k, pos, P, kv_len, d_t, d_h, d_w, eps=1e-6, theta=10000.0,
                           work=None, stream=None, fused=True, attn_chunks=1, exchange_stream=None):
    """One pass of the whole hot path over [S, H, D] q, k, v with Ulysses degree P.

    QK-norm + RoPE -> seq->head of q', k', v -> attention of each of the P
    head groups (one call per group, as each rank of a P-way group would
    issue it) -> head->seq of the output.  Returns o [S, H, D].

    fused: norm/RoPE writes q', k' straight into the head-sharded layout
      (h3attn_qk_norm_rope_seq2head) instead of norm/RoPE then seq2head.
    attn_chunks: split each group's heads into this many chunks; with an
      `exchange_stream`, the output exchange of chunk c runs on that stream
      while attention computes chunk c+1 (the result is bit-identical for any
      chunk count).  `work` may pass preallocated buffers (make_workspace).
    """
    S, H, D = q.shape
    if int(attn_chunks) != attn_chunks or attn_chunks < 1:
        raise ValueError(f"attn_chunks must be a positive integer, got {attn_chunks}")
    if work is None:
        work = make_workspace(S, H, D, P, q.device, fused=fused)
    elif not fused and not ("qr" in work and "kr" in work):
        raise ValueError("the unfused step needs a workspace from make_workspace(..., fused=False)")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    if fused:
        h3attn_qk_norm_rope_seq2head(q, k, work["qh"], work["kh"], w_q, w_k, pos, P, d_t, d_h, d_w, eps, theta,
                                     stream=stream)
    else:
        h3attn_qk_norm_rope(q, k, work["qr"], work["kr"], w_q, w_k, pos, d_t, d_h, d_w, eps, theta, stream=stream)
        h3attn_seq2head(work["qr"], work["qh"], P, stream)
        h3attn_seq2head(work["kr"], work["kh"], P, stream)
    h3attn_seq2head(v, work["vh"], P, stream)
    Hp = H // P
    if attn_chunks <= 1 and exchange_stream is None:
        for g in range(P):
            h3attn_forward(work["qh"][g], work["kh"][g], work["vh"][g], work["oh"][g], kv_len=kv_len, stream=stream)
        h3attn_head2seq(work["oh"], work["o"], P, stream)
        return work["o"]
    xs = exchange_stream if exchange_stream is not None else stream
    bounds = [round(c * Hp / attn_chunks) for c in range(attn_chunks + 1)]
    for g in range(P):
        for c in range(attn_chunks):
            j0, j1 = bounds[c], bounds[c + 1]
            if j1 <= j0:
                continue
            h3attn_forward(work["qh"][g], work["kh"][g], work["vh"][g], work["oh"][g], head_begin=j0,
                           head_count=j1 - j0, kv_len=kv_len, stream=stream)
            if xs is not stream:
                ev = torch.cuda.Event()
                ev.record(stream)
                xs.wait_event(ev)
            h3attn_head2seq_heads(work["oh"][g], work["o"], P, g, j0, j1 - j0, stream=xs)
    if xs is not stream:
        ev = torch.cuda.Event()
        ev.record(xs)
        stream.wait_event(ev)
    return work["o"]


def make_workspace(S, H, D, P, device, fused=True):
    """Buffers for ulysses_attention_step (allocated once by the caller)."""
    e = dict(dtype=torch.bfloat16, device=device)
    w = {"qh": torch.empty((P, S, H // P, D), **e), "kh": torch.empty((P, S, H // P, D), **e),
         "vh": torch.empty((P, S, H // P, D), **e), "oh": torch.empty((P, S, H // P, D), **e),
         "o": torch.empty((S, H, D), **e)}
    if not fused:
        w["qr"] = torch.empty((S, H, D), **e)
        w["kr"] = torch.empty((S, H, D), **e)
    return w


class StepGraph:
    """One ulysses_attention_step captured as a CUDA graph.

    The step's kernels (norm/RoPE + seq2head of q and k, seq2head of v, one
    attention launch per head group, head2seq) are captured once on the given
    q, k, v, weights and positions; replay() re-runs all of them with a single
    graph launch and none of the per-call host work (argument checks, tensor
    map encoding, marshalling).  Inputs are read from the same buffers at
    every replay: write new data into them (e.g. ``step.q.copy_(x)``) before
    replaying.  Returns the same output tensor every time.
    """

    def __init__(self, q, k, v, w_q, w_k, pos, P, kv_len, d_t, d_h, d_w, eps=1e-6, theta=10000.0, fused=True):
        S, H, D = q.shape
        self.q, self.k, self.v, self.w_q, self.w_k, self.pos = q, k, v, w_q, w_k, pos
        self.work = make_workspace(S, H, D, P, q.device, fused=fused)
        args = (q, k, v, w_q, w_k, pos, P, kv_len, d_t, d_h, d_w, eps, theta)
        side = torch.cuda.Stream(q.device)
        side.wait_stream(torch.cuda.current_stream(q.device))
        with torch.cuda.stream(side):
            # one eager pass first: one-time library set-up (driver entry points,
            # shared-memory attributes, the status word's address) stays out of the graph
            ulysses_attention_step(*args, work=self.work, stream=side, fused=fused)
        side.synchronize()
        status = h3attn_get_device_status(side)
        if status != H3ATTN_OK:
            raise H3AttnError("StepGraph warm-up", status)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=side):
            self.out = ulysses_attention_step(*args, work=self.work, stream=side, fused=fused)

    def replay(self):
        """Launch the captured step on the current stream; returns the output tensor."""
        self.graph.replay()
        return self.out
