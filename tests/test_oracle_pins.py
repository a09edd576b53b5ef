"""Pins for the fp64 oracle, checked against things other than itself.

Each test ties one oracle function to a hand-worked value, a closed form, an
invariant of the mathematics, brute force on tiny inputs, or an independent
library routine (torch's fp64 CPU rms_norm / scaled_dot_product_attention).
They are chosen so that a dropped term, a wrong sign or index, or a transposed
operand in the oracle fails at least one of them.  No GPU needed.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from conftest import read_golden
from dit_sequence_attention_gb300 import synth

RNG = np.random.default_rng(1234)


# ----------------------------------------------------------------- RMSNorm
def test_rmsnorm_closed_form():
    _, rows = read_golden("rmsnorm_closed_form.txt")
    assert len(rows) == 3
    for eps, w0, w1, y0, y1 in rows:
        y = oracle.rmsnorm(np.array([[3.0, 4.0]]), np.array([w0, w1]), eps)
        np.testing.assert_allclose(y[0], [y0, y1], rtol=1e-14, atol=0)


def test_rmsnorm_unit_rms_with_unit_weight():
    x = RNG.standard_normal((37, 128)) * RNG.uniform(0.1, 10, size=(37, 1))
    y = oracle.rmsnorm(x, np.ones(128), 0.0)
    np.testing.assert_allclose(np.sqrt((y * y).mean(axis=1)), 1.0, rtol=1e-14)


def test_rmsnorm_matches_torch_fp64():
    x = RNG.standard_normal((5, 7, 64))
    w = 1 + 0.1 * RNG.standard_normal(64)
    for eps in (1e-6, 0.5):
        ref = F.rms_norm(torch.from_numpy(x), (64,), torch.from_numpy(w), eps).numpy()
        np.testing.assert_allclose(oracle.rmsnorm(x, w, eps), ref, rtol=1e-13, atol=1e-15)


# -------------------------------------------------------------------- RoPE
def test_rope_worked_example():
    g, _ = read_golden("rope_worked_example.txt")
    D = int(g["D"][0])
    d_t, d_h, d_w = (int(v) for v in g["split"])
    x = np.array(g["x"]).reshape(1, 1, D)
    pos = np.array([g["pos"]], dtype=np.int32)
    y = oracle.rope(x, pos, d_t, d_h, d_w, g["theta"][0])
    np.testing.assert_allclose(y.reshape(-1), g["y"], rtol=0, atol=1e-15)


def test_norm_rope_worked_example():
    """QK-norm (weight applied to the normalised value) and then RoPE, against a
    hand-worked case whose weights differ inside each rotation pair, so that
    rotating before weighting, or weighting after the rotation, fails."""
    g, _ = read_golden("norm_rope_worked_example.txt")
    D = int(g["D"][0])
    d_t, d_h, d_w = (int(v) for v in g["split"])
    x = np.array(g["x"]).reshape(1, 1, D)
    w = np.array(g["w"])
    pos = np.array([g["pos"]], dtype=np.int32)
    for eps_key, y_key in (("eps_half", "y_eps_half"), ("eps_zero", "y_eps_zero")):
        y = oracle.norm_rope(x, w, pos, g[eps_key][0], d_t, d_h, d_w, g["theta"][0])
        np.testing.assert_allclose(y.reshape(-1), g[y_key], rtol=0, atol=1e-14)


def test_rope_zero_position_is_identity():
    x = RNG.standard_normal((9, 3, 128))
    pos = np.zeros((9, 3), dtype=np.int32)
    np.testing.assert_array_equal(oracle.rope(x, pos, 32, 48, 48), x)


def test_rope_preserves_pair_norms():
    x = RNG.standard_normal((11, 2, 128))
    pos = RNG.integers(0, 1000, size=(11, 3)).astype(np.int32)
    y = oracle.rope(x, pos, 32, 48, 48)
    nx = np.hypot(x[..., 0::2], x[..., 1::2])
    ny = np.hypot(y[..., 0::2], y[..., 1::2])
    np.testing.assert_allclose(ny, nx, rtol=1e-13)
    assert not np.allclose(y, x)


def test_rope_relative_position_property():
    """q'(p + c) . k'(r + c) == q'(p) . k'(r) for any constant shift c of all three axes."""
    S, H, D = 8, 2, 64
    q = RNG.standard_normal((S, H, D))
    k = RNG.standard_normal((S, H, D))
    pos = RNG.integers(0, 50, size=(S, 3)).astype(np.int32)
    shift = np.array([[7, -3, 11]], dtype=np.int32)
    def dots(p):
        qr = oracle.rope(q, p, 16, 24, 24)
        kr = oracle.rope(k, p, 16, 24, 24)
        return np.einsum("shd,thd->hst", qr, kr)
    np.testing.assert_allclose(dots(pos + shift), dots(pos), rtol=1e-11, atol=1e-11)
    # A shift on one axis alone changes the t-slice contribution only through
    # relative positions too, but a shift of ONE token's position must change it.
    pos2 = pos.copy()
    pos2[0, 1] += 1
    assert not np.allclose(dots(pos2), dots(pos))


def test_rope_axis_slices_use_their_own_positions():
    """Moving only the h position must leave the t and w slices untouched."""
    x = RNG.standard_normal((1, 1, 128))
    a = oracle.rope(x, np.array([[3, 5, 7]], np.int32), 32, 48, 48)
    b = oracle.rope(x, np.array([[3, 9, 7]], np.int32), 32, 48, 48)
    np.testing.assert_array_equal(a[..., :32], b[..., :32])
    np.testing.assert_array_equal(a[..., 80:], b[..., 80:])
    assert not np.allclose(a[..., 32:80], b[..., 32:80])


def test_rope_rotate_half_is_a_permutation_of_interleaved():
    """The non-interleaved pairing flag is the interleaved one under a dim permutation."""
    D, split = 16, (4, 4, 8)
    x = RNG.standard_normal((5, 2, D))
    pos = RNG.integers(0, 20, size=(5, 3)).astype(np.int32)
    perm = []
    off = 0
    for da in split:            # interleaved slot (2i, 2i+1) <- half-split (i, i + da/2)
        for i in range(da // 2):
            perm += [off + i, off + i + da // 2]
        off += da
    perm = np.array(perm)
    y_half = oracle.rope(x, pos, *split, interleaved=False)
    y_int = oracle.rope(x[..., perm], pos, *split, interleaved=True)
    np.testing.assert_allclose(y_half[..., perm], y_int, rtol=0, atol=1e-15)


# --------------------------------------------------------------- attention
def test_attention_worked_example():
    g, _ = read_golden("attention_worked_example.txt")
    q = np.array(g["q"]).reshape(1, 1, 2)
    k = np.array(g["k"]).reshape(3, 1, 2)
    v = np.array(g["v"]).reshape(3, 1, 2)
    o = oracle.attention(q, k, v, kv_len=int(g["kv_len"][0]))
    np.testing.assert_allclose(o.reshape(-1), g["o"], rtol=1e-14)


def test_attention_matches_torch_sdpa_fp64_with_key_mask():
    S, H, D, kv = 70, 3, 32, 53
    q, k, v = (RNG.standard_normal((S, H, D)) for _ in range(3))
    o = oracle.attention(q, k, v, kv_len=kv)
    tq, tk, tv = (torch.from_numpy(a).permute(1, 0, 2)[None] for a in (q, k, v))
    mask = torch.zeros(S, S, dtype=torch.bool)
    mask[:, :kv] = True
    ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)[0].permute(1, 0, 2).numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-13)


def test_attention_brute_force_python_loops():
    S, H, D, kv = 6, 2, 4, 5
    q, k, v = (RNG.standard_normal((S, H, D)) for _ in range(3))
    o = oracle.attention(q, k, v, kv_len=kv, scale=0.37)
    for h in range(H):
        for i in range(S):
            w = [math.exp(0.37 * sum(q[i, h, d] * k[j, h, d] for d in range(D))) for j in range(kv)]
            for d in range(D):
                ref = sum(w[j] * v[j, h, d] for j in range(kv)) / sum(w)
                assert abs(o[i, h, d] - ref) <= 1e-12 * (1 + abs(ref))


def test_attention_uniform_values_returns_that_value():
    S, H, D = 40, 2, 16
    q, k = RNG.standard_normal((S, H, D)) * 3, RNG.standard_normal((S, H, D)) * 3
    row = RNG.standard_normal((1, H, D))
    v = np.repeat(row, S, axis=0)
    o = oracle.attention(q, k, v, kv_len=31)
    np.testing.assert_allclose(o, np.repeat(row, S, axis=0), rtol=1e-13, atol=1e-14)


def test_attention_single_valid_key_returns_v0():
    S, H, D = 12, 2, 8
    q, k, v = (RNG.standard_normal((S, H, D)) for _ in range(3))
    o = oracle.attention(q, k, v, kv_len=1)
    np.testing.assert_array_equal(o, np.repeat(v[:1], S, axis=0))


def test_attention_zero_query_returns_mean_of_valid_values():
    S, H, D, kv = 20, 3, 8, 13
    k, v = RNG.standard_normal((S, H, D)), RNG.standard_normal((S, H, D))
    o = oracle.attention(np.zeros((4, H, D)), k, v, kv_len=kv)
    np.testing.assert_allclose(o, np.repeat(v[:kv].mean(axis=0, keepdims=True), 4, axis=0),
                               rtol=1e-13, atol=1e-15)


def test_attention_key_value_permutation_invariance():
    S, H, D = 33, 2, 16
    q, k, v = (RNG.standard_normal((S, H, D)) for _ in range(3))
    perm = RNG.permutation(S)
    np.testing.assert_allclose(oracle.attention(q, k[perm], v[perm]), oracle.attention(q, k, v),
                               rtol=1e-12, atol=1e-14)


def test_attention_masked_keys_are_ignored_even_if_nan():
    S, H, D, kv = 48, 2, 16, 29
    q, k, v = (RNG.standard_normal((S, H, D)) for _ in range(3))
    o = oracle.attention(q, k, v, kv_len=kv)
    k2, v2 = k.copy(), v.copy()
    k2[kv:] = np.nan
    v2[kv:] = np.nan
    np.testing.assert_array_equal(oracle.attention(q, k2, v2, kv_len=kv), o)
    # padded + masked equals unpadded
    np.testing.assert_allclose(oracle.attention(q, k[:kv], v[:kv]), o, rtol=1e-14, atol=0)


def test_attention_head_subsets_equal_all_heads():
    S, H, D = 24, 8, 16
    q, k, v = (RNG.standard_normal((S, H, D)) for _ in range(3))
    full = oracle.attention(q, k, v)
    for g in range(4):
        sl = slice(2 * g, 2 * g + 2)
        np.testing.assert_array_equal(oracle.attention(q[:, sl], k[:, sl], v[:, sl]), full[:, sl])


def test_attention_row_subset_equals_full_rows():
    S, H, D = 30, 2, 8
    q, k, v = (RNG.standard_normal((S, H, D)) for _ in range(3))
    rows = np.array([0, 7, 29])
    np.testing.assert_array_equal(oracle.attention(q[rows], k, v), oracle.attention(q, k, v)[rows])


# ------------------------------------------------------------------ layout
@pytest.mark.parametrize("P", [1, 2, 4, 7, 8])
def test_layout_matches_numpy_transpose_and_roundtrips(P):
    S, H, D = 56, 56, 8
    x = RNG.integers(0, 2 ** 16, size=(S, H, D), dtype=np.uint16)
    out = oracle.seq2head(x, P)
    ref = x.reshape(S, P, H // P, D).transpose(1, 0, 2, 3)
    np.testing.assert_array_equal(out, ref)
    np.testing.assert_array_equal(oracle.head2seq(out, P), x)


def test_layout_shard_view_per_element():
    """Rank r's shard row i, head g*H/P + j lands at group g, row r*S/P + i, slot j."""
    S, H, D, P = 12, 6, 2, 3
    x = RNG.integers(0, 2 ** 16, size=(S, H, D), dtype=np.uint16)
    out = oracle.seq2head(x, P)
    shards = x.reshape(P, S // P, H, D)
    for r in range(P):
        for i in range(S // P):
            for g in range(P):
                for j in range(H // P):
                    np.testing.assert_array_equal(out[g, r * (S // P) + i, j],
                                                  shards[r, i, g * (H // P) + j])


# ----------------------------------------------------------- synthetic data
def test_workload_shapes_and_positions():
    for name, S_v, S in (("tiny", 256, 256), ("c2", 4040, 4096), ("480p", 50912, 51200),
                         ("480p_p7", 50912, 53760), ("1080p", 262112, 262144)):
        w = synth.WORKLOADS[name]
        assert (w.S_v, w.S) == (S_v, S)
        assert w.S % 512 == 0 or name == "tiny"   # tiny: 256 tokens, no padding
        assert sum(w.rope_split) == w.D
    w = synth.WORKLOADS["tiny"]
    pos = synth.packed_positions(w)
    assert pos.shape == (256, 3)
    np.testing.assert_array_equal(pos[:16, 0], np.arange(16))
    assert (pos[:16, 1:] == 0).all()
    assert tuple(pos[16]) == (0, 0, 0) and tuple(pos[17]) == (0, 0, 1)
    assert tuple(pos[16 + 60]) == (1, 0, 0) and tuple(pos[-1]) == (3, 5, 9)
    assert synth.WORKLOADS["480p_p7"].S % 7 == 0


def test_seeded_inputs_are_reproducible():
    a = synth.randn_bf16((4, 3, 8), 7)
    b = synth.randn_bf16((4, 3, 8), 7)
    assert torch.equal(a, b) and a.dtype == torch.bfloat16
    wq, wk = synth.norm_weights(64)
    assert wq.shape == (64,) and not torch.equal(wq, wk)


# ------------------------------------------------- fp8 QKV projection (all-gather variant)
def test_e4m3_decode_golden():
    import os
    from conftest import GOLDEN
    for line in open(os.path.join(GOLDEN, "e4m3_decode.txt")):
        line = line.split("#", 1)[0].split()
        if len(line) == 2:
            assert oracle.e4m3_decode(int(line[0], 16)) == float(line[1]), line
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))


def test_e4m3_decode_matches_torch_float8_for_all_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_decode(c) for c in range(256)])
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def _fp8_codes(shape, seed, std):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_qkv_proj_matches_numpy_matmul_of_decoded_values():
    n, hidden, inner = 5, 96, 32
    x, w = _fp8_codes((n, hidden), 1, 1.0), _fp8_codes((3 * inner, hidden), 2, 4.0)
    table = np.array([oracle.e4m3_decode(c) for c in range(256)])
    ref = (table[x] @ table[w].T) * 0.125
    got = oracle.qkv_proj_fp8(x, w, 0.125, inner, 1, 0)
    np.testing.assert_allclose(got.reshape(n, 3 * inner), ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("P", [2, 4, 7, 8])
def test_qkv_proj_rank_slices_are_the_columns_of_the_full_projection(P):
    n, hidden, inner = 3, 64, 56
    x, w = _fp8_codes((n, hidden), 3, 1.0), _fp8_codes((3 * inner, hidden), 4, 2.0)
    full = oracle.qkv_proj_fp8(x, w, 0.5, inner, 1, 0)          # [n, 3, inner]
    parts = np.concatenate([oracle.qkv_proj_fp8(x, w, 0.5, inner, P, r) for r in range(P)], axis=2)
    np.testing.assert_array_equal(parts, full)


def test_qkv_proj_brute_force_python_loops():
    n, hidden, inner, P, rank = 2, 8, 4, 2, 1
    x, w = _fp8_codes((n, hidden), 5, 1.0), _fp8_codes((3 * inner, hidden), 6, 1.0)
    got = oracle.qkv_proj_fp8(x, w, 2.0, inner, P, rank)
    for r in range(n):
        for part in range(3):
            for c in range(inner // P):
                row = part * inner + rank * (inner // P) + c
                ref = 2.0 * sum(oracle.e4m3_decode(x[r, e]) * oracle.e4m3_decode(w[row, e]) for e in range(hidden))
                assert got[r, part, c] == pytest.approx(ref, rel=1e-14, abs=1e-14)
