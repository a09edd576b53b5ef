"""The C-ABI library builds, loads without a GPU and exports every symbol that
include/h3attn.h declares; host-side argument checks run before any CUDA call.
No GPU needed (no compute call is made)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from dit_sequence_attention_gb300 import build
    build.build()
    import dit_sequence_attention_gb300 as h3
    return h3.load_library()


def declared_functions():
    with open(os.path.join(ROOT, "include", "h3attn.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(h3attn_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("h3attn_qk_norm_rope", "h3attn_forward", "h3attn_seq2head", "h3attn_head2seq",
                     "h3attn_get_device_status", "h3attn_strerror"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    import dit_sequence_attention_gb300 as h3
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared but not exported"
        assert name in h3.SIGNATURES, f"{name} has no Python binding"


def test_no_undeclared_exports():
    # every exported h3attn_* symbol must be declared in the header
    import subprocess
    import dit_sequence_attention_gb300 as h3
    out = subprocess.run(["nm", "-D", "--defined-only", h3.library_path()], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\b(h3attn_\w+)$", out, flags=re.M))
    assert exported == set(declared_functions())


def test_version_and_strerror_need_no_gpu(lib):
    assert lib.h3attn_version() == 1
    assert lib.h3attn_strerror(0) == b"ok"
    assert b"timeout" in lib.h3attn_strerror(-5)
    assert b"index check" in lib.h3attn_strerror(-7)
    assert lib.h3attn_strerror(12345) == b"unknown status"


@pytest.fixture(scope="module")
def debug_lib():
    from dit_sequence_attention_gb300 import build
    path = build.build(debug=True)
    import dit_sequence_attention_gb300 as h3
    dl = ctypes.CDLL(path)
    for name, (res, args) in h3.SIGNATURES.items():
        getattr(dl, name).restype = res
        getattr(dl, name).argtypes = args
    return dl


def test_build_flags_tell_the_two_builds_apart(lib, debug_lib):
    import dit_sequence_attention_gb300 as h3
    assert lib.h3attn_build_flags() == 0
    assert debug_lib.h3attn_build_flags() == h3.H3ATTN_BUILD_DEBUG_CHECKS


def test_debug_build_exports_the_same_symbols(debug_lib):
    import subprocess
    from dit_sequence_attention_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB_DEBUG], capture_output=True, text=True).stdout
    assert set(re.findall(r"\b(h3attn_\w+)$", out, flags=re.M)) == set(declared_functions())


def test_bounds_selftest_refuses_without_checks_or_buffer(lib, debug_lib):
    import dit_sequence_attention_gb300 as h3
    fake = 0x10000000
    # the release build has no checks to test: refused before any CUDA call
    assert lib.h3attn_selftest_bounds(fake, 4096, None) == h3.H3ATTN_ERR_ARG
    # the debug build refuses a null, misaligned or too small buffer before any CUDA call
    assert debug_lib.h3attn_selftest_bounds(None, 4096, None) == h3.H3ATTN_ERR_ARG
    assert debug_lib.h3attn_selftest_bounds(fake + 8, 4096, None) == h3.H3ATTN_ERR_ARG
    assert debug_lib.h3attn_selftest_bounds(fake, 1008, None) == h3.H3ATTN_ERR_ARG


def test_argument_checks_run_before_any_cuda_call(lib):
    import dit_sequence_attention_gb300 as h3
    null = None
    fake = 0x10000  # aligned, never dereferenced: the checks reject the call first
    assert lib.h3attn_forward(null, fake, fake, fake, 1, 256, 4, 64, 0, 4, null, 0.0, null) == h3.H3ATTN_ERR_ARG
    assert lib.h3attn_forward(fake, fake + 0x100000, fake + 0x200000, fake + 0x300000, 1, 256, 4, 96, 0, 4,
                              null, 0.0, null) == h3.H3ATTN_ERR_SHAPE
    assert lib.h3attn_forward(fake, fake + 0x100000, fake + 0x200000, fake + 0x300000, 1, 256, 4, 64, 2, 3,
                              null, 0.0, null) == h3.H3ATTN_ERR_SHAPE
    kv = (ctypes.c_int32 * 1)(0)
    assert lib.h3attn_forward(fake, fake + 0x100000, fake + 0x200000, fake + 0x300000, 1, 256, 4, 64, 0, 4,
                              ctypes.cast(kv, ctypes.c_void_p), 0.0, null) == h3.H3ATTN_ERR_SHAPE
    assert lib.h3attn_forward(fake, fake, fake, fake, 1, 256, 4, 64, 0, 4, null, 0.0, null) == h3.H3ATTN_ERR_ALIAS
    assert lib.h3attn_forward(fake + 8, fake + 0x100000, fake + 0x200000, fake + 0x300000, 1, 256, 4, 64, 0, 4,
                              null, 0.0, null) == h3.H3ATTN_ERR_ARG
    assert lib.h3attn_seq2head(fake, fake + 0x100000, 64, 56, 128, 3, null) == h3.H3ATTN_ERR_SHAPE
    assert lib.h3attn_seq2head(fake, fake + 0x100, 64, 56, 128, 2, null) == h3.H3ATTN_ERR_ALIAS
    assert lib.h3attn_head2seq(fake, fake + 0x100000, 63, 56, 128, 2, null) == h3.H3ATTN_ERR_SHAPE
    # norm/rope: split must sum to D, even widths, eps >= 0, theta > 0
    args = [fake, fake + 0x100000, fake + 0x200000, fake + 0x300000, null, fake + 0x400000, fake + 0x500000,
            fake + 0x600000, 1, 16, 4, 64]
    f = lib.h3attn_qk_norm_rope
    assert f(*args, 16, 24, 22, 1e-6, 1e4, null) == h3.H3ATTN_ERR_SHAPE
    assert f(*args, 15, 25, 24, 1e-6, 1e4, null) == h3.H3ATTN_ERR_SHAPE
    assert f(*args, 16, 24, 24, -1.0, 1e4, null) == h3.H3ATTN_ERR_ARG
    assert f(*args, 16, 24, 24, 1e-6, 0.0, null) == h3.H3ATTN_ERR_ARG
    assert lib.h3attn_selftest_wait_timeout(0, null) == h3.H3ATTN_ERR_ARG
    g = lib.h3attn_qk_norm_rope_seq2head
    base = [fake, fake + 0x100000, fake + 0x200000, fake + 0x300000, null, fake + 0x400000, fake + 0x500000,
            fake + 0x600000]
    assert g(*base, 64, 56, 128, 3, 32, 48, 48, 1e-6, 1e4, null) == h3.H3ATTN_ERR_SHAPE      # P does not divide H
    assert g(*base, 64, 56, 128, 2, 32, 48, 46, 1e-6, 1e4, null) == h3.H3ATTN_ERR_SHAPE      # split != D
    assert g(fake, fake + 0x100000, fake + 0x10, fake + 0x300000, null, fake + 0x400000, fake + 0x500000,
             fake + 0x600000, 64, 56, 128, 2, 32, 48, 48, 1e-6, 1e4, null) == h3.H3ATTN_ERR_ALIAS  # out overlaps q
    # the head-group reciprocal of the sharded store is exact only below 2^16 heads
    assert g(*base, 2, 65536, 64, 2, 16, 24, 24, 1e-6, 1e4, null) == h3.H3ATTN_ERR_SHAPE
    assert f(fake, fake + 0x10000000, fake + 0x20000000, fake + 0x30000000, null, fake + 0x40000000,
             fake + 0x50000000, fake + 0x60000000, 1, 2, 65536, 64, 16, 24, 24, 1e-6, 1e4, null) == h3.H3ATTN_ERR_SHAPE
    f2 = lib.h3attn_head2seq_heads
    assert f2(fake, fake + 0x1000000, 64, 56, 128, 2, 2, 0, 1, null) == h3.H3ATTN_ERR_SHAPE   # group >= P
    assert f2(fake, fake + 0x1000000, 64, 56, 128, 2, 1, 20, 9, null) == h3.H3ATTN_ERR_SHAPE  # past H/P
    assert f2(fake, fake + 0x100, 64, 56, 128, 2, 1, 0, 4, null) == h3.H3ATTN_ERR_ALIAS


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import dit_sequence_attention_gb300 as h3
    missing = str(tmp_path / "missing.so")
    monkeypatch.setattr(h3, "_libs", {})
    monkeypatch.setattr(h3, "_LIB_PATHS", {False: missing, True: missing})
    for debug in (False, True):
        monkeypatch.setattr(h3, "_debug", debug)
        with pytest.raises(RuntimeError, match="not built"):
            h3.load_library()


def test_header_compiles_as_c_and_the_abi_links_from_c(lib, tmp_path):
    """A C99 program includes include/h3attn.h, links libh3attn.so and calls
    the entry points that need no GPU (version, strings, flags, argument
    checks that refuse a call before any CUDA work)."""
    import shutil
    import subprocess
    import dit_sequence_attention_gb300 as h3
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(h3.library_path())
    exe = str(tmp_path / "abi_from_c")
    src = os.path.join(ROOT, "tests", "c", "abi_from_c.c")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), src,
                        "-o", exe, "-L", libdir, "-l:libh3attn.so", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert "abi_from_c ok" in r.stdout


def test_empty_and_oversized_inputs_are_refused_before_any_cuda_call(lib):
    """Empty sizes (S, B, H or a head count of 0) and sizes past the kernels'
    index limits are H3ATTN_ERR_SHAPE; nothing is launched (no GPU needed)."""
    import dit_sequence_attention_gb300 as h3
    null = None
    a, b, c, d = 0x10000, 0x10000000, 0x20000000, 0x30000000   # aligned, never dereferenced
    SHAPE = h3.H3ATTN_ERR_SHAPE
    # attention: no rows, no batch items, no heads, an empty head range, more heads than one grid row holds
    for B, S, H, hb, hc in ((1, 0, 4, 0, 4), (0, 256, 4, 0, 4), (1, 256, 0, 0, 1), (1, 256, 4, 0, 0),
                            (1, 256, 70000, 0, 65536)):
        assert lib.h3attn_forward(a, b, c, d, B, S, H, 64, hb, hc, null, 0.0, null) == SHAPE, (B, S, H, hb, hc)
    # layout exchanges: no rows / heads, and more 16-byte vectors than a 32-bit index reaches
    assert lib.h3attn_seq2head(a, b, 0, 56, 128, 2, null) == SHAPE
    assert lib.h3attn_head2seq(a, b, 64, 0, 128, 1, null) == SHAPE
    assert lib.h3attn_seq2head(a, b, 1 << 20, 1024, 128, 2, null) == SHAPE
    assert lib.h3attn_head2seq(a, b, 1 << 20, 1024, 128, 2, null) == SHAPE
    assert lib.h3attn_head2seq_heads(a, b, 64, 56, 128, 2, 0, 0, 0, null) == SHAPE
    assert lib.h3attn_head2seq_heads(a, b, 1 << 20, 1024, 128, 2, 0, 0, 1, null) == SHAPE
    # norm/RoPE: no rows, no batch items, no heads
    norm = lib.h3attn_qk_norm_rope
    for B, S, H in ((1, 0, 4), (0, 16, 4), (1, 16, 0)):
        assert norm(a, a + 0x100000, b, b + 0x100000, null, c, c + 0x1000, d, B, S, H, 64, 16, 24, 24, 1e-6, 1e4,
                    null) == SHAPE, (B, S, H)
    assert lib.h3attn_qk_norm_rope_seq2head(a, a + 0x100000, b, b + 0x100000, null, c, c + 0x1000, d, 0, 56, 128,
                                            2, 32, 48, 48, 1e-6, 1e4, null) == SHAPE
    # projection: no rows, hidden not a multiple of 16, a rank slice not a multiple of 8 columns, rank >= P
    proj = lib.h3attn_qkv_proj_fp8
    for S, hidden, inner, P, rank in ((0, 64, 512, 2, 0), (16, 40, 512, 2, 0), (16, 64, 516, 2, 0),
                                      (16, 64, 512, 2, 2), (16, 64, 512, 0, 0)):
        assert proj(a, b, 1.0, c, c + 0x1000000, c + 0x2000000, S, hidden, inner, P, rank, null) == SHAPE, \
            (S, hidden, inner, P, rank)


def test_step_arguments_are_checked_before_any_launch():
    """A chunk count below one, or an unfused step handed the fused workspace,
    is refused before anything is allocated or launched (CPU tensors: a call
    that got as far as a kernel would fail on the device check instead)."""
    import torch
    import dit_sequence_attention_gb300 as h3
    S, H, D, P = 16, 4, 64, 2
    q = k = v = torch.zeros((S, H, D), dtype=torch.bfloat16)
    w = torch.ones(D)
    pos = torch.zeros((S, 3), dtype=torch.int32)
    for chunks in (0, -1, 1.5):
        with pytest.raises(ValueError, match="attn_chunks"):
            h3.ulysses_attention_step(q, k, v, w, w, pos, P, S, 16, 24, 24, attn_chunks=chunks,
                                      exchange_stream=object())
    fused_work = {name: None for name in ("qh", "kh", "vh", "oh", "o")}
    with pytest.raises(ValueError, match="unfused"):
        h3.ulysses_attention_step(q, k, v, w, w, pos, P, S, 16, 24, 24, work=fused_work, fused=False)
