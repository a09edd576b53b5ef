"""Out-of-bounds write checks without a sanitizer: every output buffer is the
middle of a larger allocation whose guard bands (and, for head-range calls,
the heads outside the range) are filled with a sentinel bit pattern; after the
call the sentinel must be intact.  Ragged sizes exercise every tail path."""
import pytest
import torch

from dit_sequence_attention_gb300 import synth

pytestmark = pytest.mark.gpu

GUARD = 4096          # elements on each side (16-byte aligned)
SENTINEL = 0x7FC1     # a NaN bit pattern for bf16


@pytest.fixture(scope="module")
def h3(cuda_device):
    from dit_sequence_attention_gb300 import build
    build.build()
    import dit_sequence_attention_gb300 as m
    m.load_library()
    return m


def guarded(shape, dev, dtype=torch.bfloat16):
    n = 1
    for d in shape:
        n *= d
    raw = torch.full((GUARD + n + GUARD,), SENTINEL, dtype=torch.int16, device=dev)
    view = raw[GUARD:GUARD + n].view(dtype).view(*shape)
    return raw, view


def assert_guards(raw):
    torch.cuda.synchronize()
    assert bool((raw[:GUARD] == SENTINEL).all()), "write before the buffer"
    assert bool((raw[-GUARD:] == SENTINEL).all()), "write after the buffer"


@pytest.mark.parametrize("S,H,D,kv,h0,hc", [(700, 3, 128, 333, 1, 1), (300, 4, 64, 300, 0, 4),
                                             (129, 2, 128, 7, 1, 1)])
def test_attention_writes_only_its_rows_and_heads(h3, cuda_device, S, H, D, kv, h0, hc):
    q, k, v = (synth.randn_bf16((S, H, D), 90 + i, cuda_device) for i in range(3))
    raw, o = guarded((S, H, D), cuda_device)
    h3.h3attn_forward(q, k, v, o, head_begin=h0, head_count=hc, kv_len=kv)
    assert h3.h3attn_get_device_status() == 0
    assert_guards(raw)
    inside = o[:, h0:h0 + hc]
    assert not torch.isnan(inside.float()).any()
    outside = torch.cat([o[:, :h0], o[:, h0 + hc:]], dim=1)
    assert bool((outside.contiguous().view(torch.int16) == SENTINEL).all())


@pytest.mark.parametrize("S,D", [(37, 64), (301, 128)])
def test_norm_rope_stays_in_bounds(h3, cuda_device, S, D):
    H = 8
    split = (16, 24, 24) if D == 64 else (32, 48, 48)
    q, k = synth.randn_bf16((S, H, D), 1, cuda_device), synth.randn_bf16((S, H, D), 2, cuda_device)
    wq, wk = (t.to(cuda_device) for t in synth.norm_weights(D))
    pos = torch.randint(0, 50, (S, 3), dtype=torch.int32,
                        generator=torch.Generator().manual_seed(62)).to(cuda_device)
    rq, qo = guarded((S, H, D), cuda_device)
    rk, ko = guarded((S, H, D), cuda_device)
    h3.h3attn_qk_norm_rope(q, k, qo, ko, wq, wk, pos, *split)
    assert_guards(rq)
    assert_guards(rk)
    assert h3.h3attn_get_device_status() == 0
    assert not torch.isnan(qo.float()).any() and not torch.isnan(ko.float()).any()


@pytest.mark.parametrize("P", [2, 7])
def test_layout_kernels_stay_in_bounds(h3, cuda_device, P):
    S, H, D = 14 * 3, 56, 128
    x = synth.randn_bf16((S, H, D), 5, cuda_device)
    raw_g, groups = guarded((P, S, H // P, D), cuda_device)
    h3.h3attn_seq2head(x, groups, P)
    assert_guards(raw_g)
    raw_o, out = guarded((S, H, D), cuda_device)
    h3.h3attn_head2seq(groups, out, P)
    assert_guards(raw_o)
    assert torch.equal(out.view(torch.int16), x.view(torch.int16))
    raw_c, chunk = guarded((S, H, D), cuda_device)
    h3.h3attn_head2seq_heads(groups[P - 1], chunk, P, P - 1, 1, 2)
    assert_guards(raw_c)
    hb = (P - 1) * (H // P) + 1
    assert torch.equal(chunk[:, hb:hb + 2].contiguous().view(torch.int16), x[:, hb:hb + 2].contiguous().view(torch.int16))
    untouched = torch.cat([chunk[:, :hb], chunk[:, hb + 2:]], dim=1)
    assert bool((untouched.contiguous().view(torch.int16) == SENTINEL).all())


def test_fused_norm_rope_seq2head_stays_in_bounds(h3, cuda_device):
    S, H, D, P = 202, 8, 128, 2
    q, k = synth.randn_bf16((S, H, D), 3, cuda_device), synth.randn_bf16((S, H, D), 4, cuda_device)
    wq, wk = (t.to(cuda_device) for t in synth.norm_weights(D))
    pos = torch.randint(0, 50, (S, 3), dtype=torch.int32,
                        generator=torch.Generator().manual_seed(63)).to(cuda_device)
    rq, qh = guarded((P, S, H // P, D), cuda_device)
    rk, kh = guarded((P, S, H // P, D), cuda_device)
    h3.h3attn_qk_norm_rope_seq2head(q, k, qh, kh, wq, wk, pos, P, 32, 48, 48)
    assert h3.h3attn_get_device_status() == 0
    assert_guards(rq)
    assert_guards(rk)
    assert not torch.isnan(qh.float()).any() and not torch.isnan(kh.float()).any()


def test_qkv_proj_stays_in_bounds(h3, cuda_device):
    S, hidden, inner, P, rank = 131, 272, 896, 7, 6
    x = synth.fp8_e4m3_codes((S, hidden), 7, 1.0, cuda_device)
    w = synth.fp8_e4m3_codes((3 * inner, hidden), 8, 2.0, cuda_device)
    raws, outs = zip(*(guarded((S, inner // P), cuda_device) for _ in range(3)))
    h3.h3attn_qkv_proj_fp8(x, w, 0.01, *outs, P, rank)
    assert h3.h3attn_get_device_status() == 0
    for r, o in zip(raws, outs):
        assert_guards(r)
        assert not torch.isnan(o.float()).any()
