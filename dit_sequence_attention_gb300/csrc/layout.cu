// layout.cu -- Ulysses layout exchanges as single-GPU permutation kernels.
//
// "buqi-minimax-h3-multigpu" README, "How it works": per-token work runs on a
// sequence-sharded layout (rank r holds rows [r*S/P, (r+1)*S/P) of every
// head), attention on a head-sharded one (group g holds every row of heads
// [g*H/P, (g+1)*H/P)).  On one GPU the P shards are one [S][H][D] tensor, so
// the exchange is a regrouping of whole head rows:
//     seq2head: [S][H][D]      -> [P][S][H/P][D]
//     head2seq: [P][S][H/P][D] -> [S][H][D]
// A head row is D contiguous bf16 (128 or 256 bytes) on both sides, so no
// shared-memory transpose is needed: every thread moves 16-byte vectors, the
// read side and the write side are both fully coalesced (runs of H/P rows of
// the destination are contiguous), and each thread keeps 4 vectors in flight.
// The kernels are HBM-bound: 2 * S * H * D * 2 bytes per tensor.
#include <cstdint>

#include "h3_device.cuh"
#include "h3_internal.h"

namespace h3 {

constexpr int kLayoutThreads = 256;
constexpr int kLayoutUnroll = 4;

// seq2head: index the SOURCE (coalesced reads), scatter rows to their group.
__global__ void __launch_bounds__(kLayoutThreads) seq2head_kernel(const uint4* __restrict__ in,
                                                                  uint4* __restrict__ out, uint32_t S,
                                                                  uint32_t H, uint32_t Hp, uint32_t vpr_log2,
                                                                  uint32_t total) {
    const uint32_t base = blockIdx.x * (kLayoutThreads * kLayoutUnroll) + threadIdx.x;
    uint4 v[kLayoutUnroll];
    uint32_t dst[kLayoutUnroll];
#pragma unroll
    for (int u = 0; u < kLayoutUnroll; ++u) {
        const uint32_t i = base + u * kLayoutThreads;
        if (i < total) {
            v[u] = __ldcs(in + i);
            const uint32_t part = i & ((1u << vpr_log2) - 1u);
            const uint32_t row = i >> vpr_log2;  // s * H + h
            const uint32_t s = row / H, h = row - s * H;
            const uint32_t g = h / Hp, j = h - g * Hp;
            dst[u] = (((g * S + s) * Hp + j) << vpr_log2) + part;
        }
    }
#pragma unroll
    for (int u = 0; u < kLayoutUnroll; ++u) {
        const uint32_t i = base + u * kLayoutThreads;
        if (i < total) __stcs(out + dst[u], v[u]);
    }
}

// head2seq: index the DESTINATION (coalesced writes), gather rows from groups.
__global__ void __launch_bounds__(kLayoutThreads) head2seq_kernel(const uint4* __restrict__ in,
                                                                  uint4* __restrict__ out, uint32_t S,
                                                                  uint32_t H, uint32_t Hp, uint32_t vpr_log2,
                                                                  uint32_t total) {
    const uint32_t base = blockIdx.x * (kLayoutThreads * kLayoutUnroll) + threadIdx.x;
    uint4 v[kLayoutUnroll];
#pragma unroll
    for (int u = 0; u < kLayoutUnroll; ++u) {
        const uint32_t i = base + u * kLayoutThreads;
        if (i < total) {
            const uint32_t part = i & ((1u << vpr_log2) - 1u);
            const uint32_t row = i >> vpr_log2;  // s * H + h of the destination
            const uint32_t s = row / H, h = row - s * H;
            const uint32_t g = h / Hp, j = h - g * Hp;
            v[u] = __ldcs(in + ((((g * S + s) * Hp + j) << vpr_log2) + part));
        }
    }
#pragma unroll
    for (int u = 0; u < kLayoutUnroll; ++u) {
        const uint32_t i = base + u * kLayoutThreads;
        if (i < total) __stcs(out + i, v[u]);
    }
}

// head2seq for a chunk of one group's heads: group g's buffer [S][H/P][D],
// heads [j0, j0 + jc) -> out[s][g*(H/P) + j].  Used to overlap the output
// exchange of one head chunk with the attention of the next.
__global__ void __launch_bounds__(kLayoutThreads) head2seq_heads_kernel(const uint4* __restrict__ in,
                                                                        uint4* __restrict__ out, uint32_t H,
                                                                        uint32_t Hp, uint32_t hbase, uint32_t j0,
                                                                        uint32_t jc, uint32_t vpr_log2,
                                                                        uint32_t total) {
    const uint32_t base = blockIdx.x * (kLayoutThreads * kLayoutUnroll) + threadIdx.x;
    uint4 v[kLayoutUnroll];
#pragma unroll
    for (int u = 0; u < kLayoutUnroll; ++u) {
        const uint32_t i = base + u * kLayoutThreads;
        if (i < total) {
            const uint32_t part = i & ((1u << vpr_log2) - 1u);
            const uint32_t rest = i >> vpr_log2;  // s * jc + jj
            const uint32_t s = rest / jc, jj = rest - s * jc;
            v[u] = __ldcs(in + (((s * Hp + j0 + jj) << vpr_log2) + part));
        }
    }
#pragma unroll
    for (int u = 0; u < kLayoutUnroll; ++u) {
        const uint32_t i = base + u * kLayoutThreads;
        if (i < total) {
            const uint32_t part = i & ((1u << vpr_log2) - 1u);
            const uint32_t rest = i >> vpr_log2;
            const uint32_t s = rest / jc, jj = rest - s * jc;
            __stcs(out + (((s * H + hbase + j0 + jj) << vpr_log2) + part), v[u]);
        }
    }
}

int launch_head2seq_heads(const void* in_group, void* out, int S, int H, int D, int P, int g, int j0, int jc,
                          cudaStream_t stream) {
    const uint32_t vpr_log2 = (D == 128) ? 4u : 3u;
    const uint64_t total64 = static_cast<uint64_t>(S) * jc * (static_cast<uint64_t>(D) / 8);
    if (total64 == 0) return H3ATTN_OK;
    const uint32_t total = static_cast<uint32_t>(total64);
    const uint32_t per_block = kLayoutThreads * kLayoutUnroll;
    const uint32_t Hp = static_cast<uint32_t>(H / P);
    head2seq_heads_kernel<<<(total + per_block - 1) / per_block, kLayoutThreads, 0, stream>>>(
        static_cast<const uint4*>(in_group), static_cast<uint4*>(out), H, Hp, g * Hp, j0, jc, vpr_log2, total);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? H3ATTN_OK : cuda_fail(e);
}

static int launch_layout(bool to_heads, const void* in, void* out, int S, int H, int D, int P,
                         cudaStream_t stream) {
    const uint32_t vpr_log2 = (D == 128) ? 4u : 3u;  // 16-byte vectors per head row
    const uint64_t total64 = static_cast<uint64_t>(S) * H * (static_cast<uint64_t>(D) / 8);
    if (total64 == 0) return H3ATTN_OK;
    const uint32_t total = static_cast<uint32_t>(total64);
    const uint32_t per_block = kLayoutThreads * kLayoutUnroll;
    const uint32_t blocks = (total + per_block - 1) / per_block;
    if (to_heads)
        seq2head_kernel<<<blocks, kLayoutThreads, 0, stream>>>(static_cast<const uint4*>(in), static_cast<uint4*>(out),
                                                               S, H, H / P, vpr_log2, total);
    else
        head2seq_kernel<<<blocks, kLayoutThreads, 0, stream>>>(static_cast<const uint4*>(in), static_cast<uint4*>(out),
                                                               S, H, H / P, vpr_log2, total);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? H3ATTN_OK : cuda_fail(e);
}

int launch_seq2head(const void* in, void* out, int S, int H, int D, int P, cudaStream_t stream) {
    return launch_layout(true, in, out, S, H, D, P, stream);
}

int launch_head2seq(const void* in, void* out, int S, int H, int D, int P, cudaStream_t stream) {
    return launch_layout(false, in, out, S, H, D, P, stream);
}

}  // namespace h3
