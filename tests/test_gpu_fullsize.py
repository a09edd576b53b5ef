"""Full-size GPU parity at the benchmark's own sizes and launch configuration.

480p (51,200 tokens, 56 x 128) through the exact bench step (QK-norm+RoPE ->
seq2head P=2 -> two 28-head attention launches -> head2seq), compared with
the fp64 oracle on 4 sampled heads x 512 sampled query rows (the oracle
computes each sampled row against every valid key); the Ulysses split at P in {2, 4, 7, 8}
compared bit for bit with one all-heads call, and the permutations bit for
bit with the oracle's index formula; 1080p (262,144 tokens) through the same
step on 4 sampled heads x 512 sampled query rows.
Inputs are seeded draws on the device (torch's CUDA generator); no oracle
input comes from the library's kernels.
"""
import numpy as np
import pytest
import torch

import oracle
from dit_sequence_attention_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

ATTN_TOL = 2e-2


@pytest.fixture(scope="module")
def h3(cuda_device):
    from dit_sequence_attention_gb300 import build
    build.build()
    import dit_sequence_attention_gb300 as m
    m.load_library()
    return m


def _inputs(w, dev):
    q, k, v = (synth.randn_bf16((w.S, w.H, w.D), seed, dev, zero_rows_from=w.S_v)
               for seed in (synth.SEED_Q, synth.SEED_K, synth.SEED_V))
    wq, wk = synth.norm_weights(w.D)
    pos = synth.packed_positions(w)
    return q, k, v, wq, wk, pos


def _oracle_rows(w, q, k, v, wq, wk, pos, heads, rows):
    """fp64 oracle for the sampled (rows, heads): norm+RoPE of those q rows and of
    every key of those heads, then attention over the valid keys."""
    heads = np.asarray(heads)
    qs = oracle.bf16_to_f64(q[torch.as_tensor(rows, device=q.device)][:, heads])
    ks = oracle.bf16_to_f64(k[:, heads])
    vs = oracle.bf16_to_f64(v[:, heads])
    qr = oracle.norm_rope(qs, wq.double().numpy(), pos[rows], w.eps, *w.rope_split, w.theta)
    kr = oracle.norm_rope(ks, wk.double().numpy(), pos, w.eps, *w.rope_split, w.theta)
    return oracle.attention(qr, kr, vs, kv_len=w.S_v)


def _sample_rows_with_edges(w, n, seed):
    """n distinct query rows: the edges that matter (first rows, both sides of
    256-row query blocks and of the sequence middle, the audio/video boundary,
    the last valid rows, padding rows) plus uniformly drawn ones."""
    fixed = [0, 1, 255, 256, w.n_audio - 2, w.n_audio - 1, w.n_audio, w.n_audio + 1, w.S // 2 - 1, w.S // 2,
             w.S_v - 2, w.S_v - 1, w.S_v, w.S - 1]
    rng = np.random.default_rng(seed)
    drawn = rng.choice(w.S, n + len(fixed), replace=False)
    sampled = drawn[~np.isin(drawn, fixed)][: n - len(fixed)]           # random order kept: no bias
    rows = np.sort(np.concatenate([sampled, fixed]))
    assert len(rows) == n and len(np.unique(rows)) == n
    return rows


def test_480p_bench_step_matches_oracle_on_sampled_rows(h3, cuda_device):
    """480p through the bench's own step on 4 sampled heads (two per head
    group, the first and the last among them) x 512 sampled query rows."""
    w = synth.WORKLOADS["480p"]
    q, k, v, wq, wk, pos = _inputs(w, cuda_device)
    dev = cuda_device
    o = h3.ulysses_attention_step(q, k, v, wq.to(dev), wk.to(dev), torch.from_numpy(pos).to(dev), 2, w.S_v,
                                  *w.rope_split, w.eps, w.theta)
    assert h3.h3attn_get_device_status() == 0
    heads = [0, 27, 28, 55]
    rows = _sample_rows_with_edges(w, 512, 5)
    ref = _oracle_rows(w, q, k, v, wq, wk, pos, heads, rows)
    got = o[torch.as_tensor(rows, device=dev)][:, heads].float().cpu().numpy()
    err = np.abs(got - ref).max(axis=(0, 2)) / np.abs(ref).max(axis=(0, 2))
    assert np.all(err <= ATTN_TOL), f"per-head rel err {err}"


@pytest.mark.parametrize("P", [2, 4, 7, 8])
def test_480p_ulysses_split_is_bit_identical(h3, cuda_device, P):
    w = synth.WORKLOADS["480p_p7" if P == 7 else "480p"]
    dev = cuda_device
    q, k, v, wq, wk, pos = _inputs(w, dev)
    qr, kr = torch.empty_like(q), torch.empty_like(k)
    h3.h3attn_qk_norm_rope(q, k, qr, kr, wq.to(dev), wk.to(dev), torch.from_numpy(pos).to(dev), *w.rope_split,
                           w.eps, w.theta)
    # single all-heads call on the sequence-major tensors
    o_all = torch.empty_like(q)
    h3.h3attn_forward(qr, kr, v, o_all, kv_len=w.S_v)
    # Ulysses: seq2head -> one call per head group -> head2seq
    work = h3.make_workspace(w.S, w.H, w.D, P, dev)
    h3.h3attn_seq2head(qr, work["qh"], P)
    h3.h3attn_seq2head(kr, work["kh"], P)
    h3.h3attn_seq2head(v, work["vh"], P)
    for g in range(P):
        h3.h3attn_forward(work["qh"][g], work["kh"][g], work["vh"][g], work["oh"][g], kv_len=w.S_v)
    h3.h3attn_head2seq(work["oh"], work["o"], P)
    assert h3.h3attn_get_device_status() == 0
    assert torch.equal(work["o"].view(torch.int16), o_all.view(torch.int16))
    # the permutation itself, bit for bit against the oracle's index formula
    np.testing.assert_array_equal(oracle.bf16_bits(work["vh"]), oracle.seq2head(oracle.bf16_bits(v), P))
    back = torch.empty_like(v)
    h3.h3attn_head2seq(work["vh"], back, P)
    assert torch.equal(back.view(torch.int16), v.view(torch.int16))


def test_1080p_bench_step_matches_oracle_on_sampled_rows(h3, cuda_device):
    """1080p through the bench's own step (fused QK-norm+RoPE+seq2head, P = 2,
    two 28-head attention launches, head2seq) on 4 sampled heads -- two from
    each head group, including the first and the last -- x 512 sampled query
    rows: the audio/video boundary, the last valid row, padding rows and rows
    at both edges of 256-row query blocks among them."""
    w = synth.WORKLOADS["1080p"]
    dev = cuda_device
    q, k, v, wq, wk, pos = _inputs(w, dev)
    o = h3.ulysses_attention_step(q, k, v, wq.to(dev), wk.to(dev), torch.from_numpy(pos).to(dev), 2, w.S_v,
                                  *w.rope_split, w.eps, w.theta)
    assert h3.h3attn_get_device_status() == 0
    heads = [0, 27, 28, 55]
    rows = _sample_rows_with_edges(w, 512, 9)
    ref = _oracle_rows(w, q, k, v, wq, wk, pos, heads, rows)
    got = o[torch.as_tensor(rows, device=dev)][:, heads].float().cpu().numpy()
    err = np.abs(got - ref).max(axis=(0, 2)) / np.abs(ref).max(axis=(0, 2))
    assert np.all(err <= ATTN_TOL), f"per-head rel err {err}"
