"""The debug-check build (libh3attn_debug.so): the same kernels, each checking
its computed global indices before the access.

On valid inputs no check may fire and every result must be bit-identical to
the release build (the checks change no arithmetic).  The bounds self-test
tells the seq2head kernel that its output is one vector shorter than the
buffer really is, so the kernel's own check must refuse exactly that store and
report it -- while every access, refused or not, stays inside the buffer."""
import pytest
import torch

from dit_sequence_attention_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h3(cuda_device):
    from dit_sequence_attention_gb300 import build
    build.build()
    build.build(debug=True)
    import dit_sequence_attention_gb300 as m
    m.use_debug_checks(False)
    m.load_library()
    yield m
    m.use_debug_checks(False)


def on_both_builds(h3, fn):
    """fn() on the release build, then on the debug build; both results, each
    required to leave the device status clean."""
    h3.use_debug_checks(False)
    rel = fn()
    assert h3.h3attn_get_device_status() == 0
    h3.use_debug_checks(True)
    try:
        assert h3.h3attn_build_flags() == h3.H3ATTN_BUILD_DEBUG_CHECKS
        dbg = fn()
        status = h3.h3attn_get_device_status()
        info = h3.h3attn_last_device_error_info()
    finally:
        h3.use_debug_checks(False)
    assert status == 0, f"debug build: status {status}, info {info:#x}"
    return rel, dbg


def bits_equal(a, b):
    return torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16))


@pytest.mark.parametrize("P", [2, 7])
def test_layout_kernels(h3, cuda_device, P):
    S, H, D = 14 * 5, 56, 128
    x = synth.randn_bf16((S, H, D), 11, cuda_device)

    def run():
        g = torch.empty((P, S, H // P, D), dtype=torch.bfloat16, device=cuda_device)
        h3.h3attn_seq2head(x, g, P)
        back = torch.empty_like(x)
        h3.h3attn_head2seq(g, back, P)
        part = torch.zeros_like(x)
        h3.h3attn_head2seq_heads(g[P - 1], part, P, P - 1, 1, 3)
        return g, back, part

    rel, dbg = on_both_builds(h3, run)
    for a, b in zip(rel, dbg):
        assert bits_equal(a, b)
    assert bits_equal(dbg[1], x)


@pytest.mark.parametrize("D,split,P", [(128, (32, 48, 48), 1), (128, (32, 48, 48), 2), (64, (16, 24, 24), 4)])
def test_norm_rope(h3, cuda_device, D, split, P):
    S, H = 301 if P == 1 else 300, 8
    q, k = synth.randn_bf16((S, H, D), 21, cuda_device), synth.randn_bf16((S, H, D), 22, cuda_device)
    wq, wk = (t.to(cuda_device) for t in synth.norm_weights(D))
    pos = torch.randint(0, 50, (S, 3), dtype=torch.int32,
                        generator=torch.Generator().manual_seed(61)).to(cuda_device)

    def run():
        dbg32 = torch.empty((2, S, H, D), dtype=torch.float32, device=cuda_device)
        if P == 1:
            qo, ko = torch.empty_like(q), torch.empty_like(k)
            h3.h3attn_qk_norm_rope(q, k, qo, ko, wq, wk, pos, *split, dbg_fp32=dbg32)
        else:
            qo = torch.empty((P, S, H // P, D), dtype=torch.bfloat16, device=cuda_device)
            ko = torch.empty_like(qo)
            h3.h3attn_qk_norm_rope_seq2head(q, k, qo, ko, wq, wk, pos, P, *split, dbg_fp32=dbg32)
        return qo, ko, dbg32

    rel, dbg = on_both_builds(h3, run)
    assert bits_equal(rel[0], dbg[0]) and bits_equal(rel[1], dbg[1])
    assert torch.equal(rel[2].view(torch.int32), dbg[2].view(torch.int32))


@pytest.mark.parametrize("S,H,D,kv,h0,hc", [(700, 3, 128, 333, 1, 2), (300, 4, 64, 300, 0, 4), (129, 2, 128, 7, 1, 1)])
def test_attention(h3, cuda_device, S, H, D, kv, h0, hc):
    q, k, v = (synth.randn_bf16((S, H, D), 31 + i, cuda_device) for i in range(3))

    def run():
        o = torch.zeros_like(q)
        h3.h3attn_forward(q, k, v, o, head_begin=h0, head_count=hc, kv_len=kv)
        return o

    rel, dbg = on_both_builds(h3, run)
    assert bits_equal(rel, dbg)


def test_attention_batch(h3, cuda_device):
    B, S, H, D = 2, 384, 2, 128
    q, k, v = (synth.randn_bf16((B, S, H, D), 41 + i, cuda_device) for i in range(3))

    def run():
        o = torch.zeros_like(q)
        h3.h3attn_forward(q, k, v, o, kv_len=[384, 200])
        return o

    rel, dbg = on_both_builds(h3, run)
    assert bits_equal(rel, dbg)


def test_qkv_proj(h3, cuda_device):
    S, hidden, inner, P, rank = 131, 272, 896, 7, 6
    x = synth.fp8_e4m3_codes((S, hidden), 51, 1.0, cuda_device)
    w = synth.fp8_e4m3_codes((3 * inner, hidden), 52, 2.0, cuda_device)

    def run():
        outs = [torch.empty((S, inner // P), dtype=torch.bfloat16, device=cuda_device) for _ in range(3)]
        h3.h3attn_qkv_proj_fp8(x, w, 0.01, *outs, P, rank)
        return outs

    rel, dbg = on_both_builds(h3, run)
    for a, b in zip(rel, dbg):
        assert bits_equal(a, b)


def test_whole_step(h3, cuda_device):
    w = synth.WORKLOADS["tiny"]
    q, k, v = (t.to(cuda_device) for t in synth.qkv(w))
    wq, wk = (t.to(cuda_device) for t in synth.norm_weights(w.D))
    pos = torch.from_numpy(synth.packed_positions(w)).to(cuda_device)

    def run():
        return h3.ulysses_attention_step(q, k, v, wq, wk, pos, 2, w.S_v, *w.rope_split, w.eps, w.theta).clone()

    rel, dbg = on_both_builds(h3, run)
    assert bits_equal(rel, dbg)


def test_bounds_check_fires_and_reports(h3, cuda_device):
    # buf[0, 512): the self-test's input, S=2 x H=2 rows of 64 bf16 = 32 vectors of 16 bytes;
    # buf[512, 1024): its output, [P=2][S=2][1][64]; the rest is spare
    buf = torch.full((2048,), 0xAB, dtype=torch.uint8, device=cuda_device)
    src = (torch.arange(512, device=cuda_device) % 251 + 1).to(torch.uint8)
    buf[:512] = src
    h3.use_debug_checks(True)
    try:
        assert h3.h3attn_get_device_status() == 0
        h3.h3attn_selftest_bounds(buf)
        status = h3.h3attn_get_device_status()
        info = h3.h3attn_last_device_error_info()
        again = h3.h3attn_get_device_status()
    finally:
        h3.use_debug_checks(False)
    assert status == h3.H3ATTN_ERR_DEVICE_BOUNDS
    # tag 5 (seq2head) << 32 | site 1 << 16 | refused output vector 31
    assert info == (5 << 32) | (1 << 16) | 31
    assert again == 0  # reading the status clears it; the context stays usable
    # the other 31 vectors hold seq2head of the input: row (s, h) -> (g = h, s)
    vin = src.view(2, 2, 8, 16)             # [s][h][vector][byte]
    want = vin.permute(1, 0, 2, 3).reshape(32, 16)
    got = buf[512:1024].view(32, 16)
    assert torch.equal(got[:31], want[:31])
    assert bool((got[31] == 0xAB).all())    # the refused store never happened
    assert bool((buf[1024:] == 0xAB).all())


def test_bounds_selftest_refused_by_release_build(h3, cuda_device):
    buf = torch.zeros(2048, dtype=torch.uint8, device=cuda_device)
    with pytest.raises(h3.H3AttnError) as e:
        h3.h3attn_selftest_bounds(buf)
    assert e.value.code == h3.H3ATTN_ERR_ARG
