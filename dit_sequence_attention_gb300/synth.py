"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds workload *shapes* and random draws only: the packed
[audio | video | pad] token layout with its (t, h, w) position triples, and
seeded N(0, 1) q/k/v plus RMSNorm weights 1 + 0.1 N(0, 1).  It contains none
of the method's arithmetic (no normalisation, rotation, softmax or layout
permutation), so both sides can import it without sharing any computation.

Workload shapes follow the packed-sequence description of the MiniMax-H3 DiT
("buqi-minimax-h3-multigpu" README, section "How it works": one packed
sequence, 56 heads) and the 512-multiple padding of the diffusers TP PR
(comment on NKI flash attention needing L % 512 == 0).  The grids are the
synthetic 480p-like and 1080p-like shapes of the benchmark contract.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

SEED_Q, SEED_K, SEED_V, SEED_W = 1, 2, 3, 4


@dataclass(frozen=True)
class Workload:
    """One packed sequence: ``n_audio`` audio tokens, then a video grid, then pad."""

    name: str
    H: int
    D: int
    frames: int
    grid_h: int
    grid_w: int
    n_audio: int
    S: int                      # padded length (keys >= S_v are masked)
    rope_split: tuple = field(default=(32, 48, 48))   # (d_t, d_h, d_w) in dims
    theta: float = 10000.0
    eps: float = 1e-6
    B: int = 1

    @property
    def n_video(self) -> int:
        return self.frames * self.grid_h * self.grid_w

    @property
    def S_v(self) -> int:
        """Number of valid (unmasked) tokens."""
        return self.n_audio + self.n_video

    def attention_flops(self, heads: int | None = None) -> float:
        """4 * S_v^2 * D per head: QK^T and PV, 2 flops per multiply-add."""
        h = self.H if heads is None else heads
        return 4.0 * float(self.S_v) ** 2 * self.D * h * self.B


WORKLOADS = {
    # 4x6x10 video grid + 16 audio tokens, no padding, 4 heads of 64.
    "tiny": Workload("tiny", H=4, D=64, frames=4, grid_h=6, grid_w=10,
                     n_audio=16, S=256, rope_split=(16, 24, 24)),
    # 8x16x30 video + 200 audio = 4040 valid, padded to 4096.
    "c2": Workload("c2", H=56, D=128, frames=8, grid_h=16, grid_w=30,
                   n_audio=200, S=4096),
    # 16x30x32 video + 992 audio = 16,352 valid, padded to 16,384: a profiling-size
    # case whose tensors (235 MB each) still exceed L2.
    "16k": Workload("16k", H=56, D=128, frames=16, grid_h=30, grid_w=32,
                    n_audio=992, S=16384),
    # 32x30x52 video + 992 audio = 50,912 valid, padded to 51,200.
    "480p": Workload("480p", H=56, D=128, frames=32, grid_h=30, grid_w=52,
                     n_audio=992, S=51200),
    # Same valid tokens, padded to 53,760 = 15 * lcm(512, 7) so seven shards divide it.
    "480p_p7": Workload("480p_p7", H=56, D=128, frames=32, grid_h=30, grid_w=52,
                        n_audio=992, S=53760),
    # 32x68x120 video + 992 audio = 262,112 valid, padded to 262,144.
    "1080p": Workload("1080p", H=56, D=128, frames=32, grid_h=68, grid_w=120,
                      n_audio=992, S=262144),
}


def packed_positions(w: Workload) -> np.ndarray:
    """int32 [S, 3] position triples for the packed sequence.

    Audio token a gets (a, 0, 0); video token (t, y, x) of the grid, enumerated
    t-major then y then x, gets (t, y, x); padding rows get (0, 0, 0).
    """
    pos = np.zeros((w.S, 3), dtype=np.int32)
    pos[: w.n_audio, 0] = np.arange(w.n_audio, dtype=np.int32)
    t, y, x = np.meshgrid(np.arange(w.frames), np.arange(w.grid_h),
                          np.arange(w.grid_w), indexing="ij")
    v0 = w.n_audio
    pos[v0: v0 + w.n_video, 0] = t.reshape(-1)
    pos[v0: v0 + w.n_video, 1] = y.reshape(-1)
    pos[v0: v0 + w.n_video, 2] = x.reshape(-1)
    return pos


def randn_bf16(shape, seed: int, device="cpu", zero_rows_from: int | None = None) -> torch.Tensor:
    """Seeded N(0, 1) draws stored as bf16.

    On CPU the draw uses torch's CPU generator; on a CUDA device it uses that
    device's generator (far faster for GB-sized tensors).  Either way the
    same (seed, device type) gives the same bits.  Rows >= ``zero_rows_from``
    along dim 0 (the padding tokens) are set to zero when given.
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    t = torch.randn(shape, generator=g, dtype=torch.float32, device=dev).to(torch.bfloat16)
    if zero_rows_from is not None:
        t[zero_rows_from:] = 0
    return t


def norm_weights(D: int, seed: int = SEED_W) -> tuple[torch.Tensor, torch.Tensor]:
    """RMSNorm weights for q and k: 1 + 0.1 N(0, 1), fp32 [D] each (CPU)."""
    g = torch.Generator()
    g.manual_seed(seed)
    w = 1.0 + 0.1 * torch.randn((2, D), generator=g, dtype=torch.float32)
    return w[0].contiguous(), w[1].contiguous()


def qkv(w: Workload, device="cpu", zero_pad=True):
    """Seeded q, k, v bf16 [S, H, D] for one batch item (pad rows zero)."""
    z = w.S_v if zero_pad else None
    shape = (w.S, w.H, w.D)
    return (randn_bf16(shape, SEED_Q, device, z),
            randn_bf16(shape, SEED_K, device, z),
            randn_bf16(shape, SEED_V, device, z))


# Hidden / projection sizes of the H3 block: hidden 5376, attention inner width
# 7168 = 56 heads x 128 ("buqi-minimax-h3-multigpu" README, "How it works").
HIDDEN, INNER = 5376, 7168


def fp8_e4m3_codes(shape, seed: int, std: float, device="cpu") -> torch.Tensor:
    """Seeded N(0, std^2) draws rounded to FP8 E4M3, returned as raw uint8 codes."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    t = torch.randn(shape, generator=g, dtype=torch.float32, device=dev) * std
    return t.to(torch.float8_e4m3fn).view(torch.uint8)
