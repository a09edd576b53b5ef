"""GPU parity of the all-gather variant's FP8 QKV projection (h3attn_qkv_proj_fp8)
against the fp64 oracle, and the row-slice equivalence the pages rely on: each
rank's projection equals the matching columns of the full projection, bit for
bit.  Tolerance: fp8 products are exact in fp32, the fp32 accumulation adds
~1e-6 relative, the bf16 output rounding adds half an ulp (2^-9 relative)."""
import numpy as np
import pytest
import torch

import oracle
from dit_sequence_attention_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h3(cuda_device):
    from dit_sequence_attention_gb300 import build
    build.build()
    import dit_sequence_attention_gb300 as m
    m.load_library()
    return m


def _run(h3, x, w, scale, P, rank):
    S = x.shape[0]
    nr = w.shape[0] // 3 // P
    outs = [torch.empty((S, nr), dtype=torch.bfloat16, device=x.device) for _ in range(3)]
    h3.h3attn_qkv_proj_fp8(x, w, scale, *outs, P, rank)
    assert h3.h3attn_get_device_status() == 0
    return outs


def _check(got_parts, ref):
    """got_parts: 3 x [n, nr] bf16 tensors; ref: [n, 3, nr] float64."""
    for part in range(3):
        got = got_parts[part].double().cpu().numpy()
        r = ref[:, part, :]
        bound = 2.0 ** -8 * np.abs(r) + 1e-5 * np.abs(r).max()
        assert np.all(np.abs(got - r) <= bound), f"part {part}: max err {np.abs(got - r).max():.3e}"


@pytest.mark.parametrize("S,hidden,inner,P,rank", [
    (300, 256, 512, 1, 0),     # ragged token tail, two N tiles per part
    (300, 256, 512, 2, 1),     # one 256-wide tile per part
    (129, 384, 512, 4, 3),     # 128-wide slice: the tile reaches into the next rank's rows
    (257, 272, 896, 7, 2),     # hidden not a multiple of 128 (zero-filled K tail)
    (200, 512, 1024, 8, 5),    # 128-wide slices
])
def test_qkv_proj_matches_oracle(h3, cuda_device, S, hidden, inner, P, rank):
    x = synth.fp8_e4m3_codes((S, hidden), 11, 1.0)
    w = synth.fp8_e4m3_codes((3 * inner, hidden), 12, 4.0)
    scale = 1.0 / (4.0 * hidden ** 0.5)
    got = _run(h3, x.to(cuda_device), w.to(cuda_device), scale, P, rank)
    ref = oracle.qkv_proj_fp8(x.numpy(), w.numpy(), scale, inner, P, rank)
    _check(got, ref)


@pytest.mark.parametrize("P", [2, 4, 7, 8])
def test_rank_slices_bit_identical_to_full_projection(h3, cuda_device, P):
    S, hidden, inner = 384, 512, synth.INNER  # inner width of H3 (56 heads x 128), small hidden
    x = synth.fp8_e4m3_codes((S, hidden), 21, 1.0, cuda_device)
    w = synth.fp8_e4m3_codes((3 * inner, hidden), 22, 4.0, cuda_device)
    full = _run(h3, x, w, 0.01, 1, 0)
    nr = inner // P
    for r in range(P):
        parts = _run(h3, x, w, 0.01, P, r)
        for part in range(3):
            assert torch.equal(parts[part].view(torch.int16),
                               full[part][:, r * nr:(r + 1) * nr].contiguous().view(torch.int16)), (P, r, part)


def test_h3_sizes_sampled_rows(h3, cuda_device):
    S, hidden, inner, P, rank = 4096, synth.HIDDEN, synth.INNER, 2, 1
    x = synth.fp8_e4m3_codes((S, hidden), 31, 1.0, cuda_device)
    w = synth.fp8_e4m3_codes((3 * inner, hidden), 32, 4.0, cuda_device)
    scale = 1.0 / (4.0 * hidden ** 0.5)
    got = _run(h3, x, w, scale, P, rank)
    rows = np.array([0, 1, 127, 128, 2047, 4094, 4095])
    ref = oracle.qkv_proj_fp8(x[torch.as_tensor(rows, device=cuda_device)].cpu().numpy(), w.cpu().numpy(), scale,
                              inner, P, rank)
    _check([g[torch.as_tensor(rows, device=cuda_device)] for g in got], ref)
