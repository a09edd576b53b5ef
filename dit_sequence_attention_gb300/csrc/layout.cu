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
// `total`: 16-byte vectors read; `out_extent`: vectors the output holds (the
// same number, except in the bounds self-test); `st`: device status word,
// used by debug-check builds only.
__global__ void __launch_bounds__(kLayoutThreads) seq2head_kernel(const uint4* __restrict__ in,
                                                                  uint4* __restrict__ out, uint32_t S,
                                                                  uint32_t H, uint32_t Hp, uint32_t vpr_log2,
                                                                  uint32_t total, uint32_t out_extent,
                                                                  DeviceStatus* st) {
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
        if (i < total && in_bounds(st, dst[u], 1, out_extent, kTagSeq2Head, 1)) __stcs(out + dst[u], v[u]);
    }
}

// head2seq: index the DESTINATION (coalesced writes), gather rows from groups.
__global__ void __launch_bounds__(kLayoutThreads) head2seq_kernel(const uint4* __restrict__ in,
                                                                  uint4* __restrict__ out, uint32_t S,
                                                                  uint32_t H, uint32_t Hp, uint32_t vpr_log2,
                                                                  uint32_t total, DeviceStatus* st) {
    const uint32_t base = blockIdx.x * (kLayoutThreads * kLayoutUnroll) + threadIdx.x;
    uint4 v[kLayoutUnroll];
    bool ok[kLayoutUnroll];
#pragma unroll
    for (int u = 0; u < kLayoutUnroll; ++u) {
        const uint32_t i = base + u * kLayoutThreads;
        ok[u] = false;
        if (i < total) {
            const uint32_t part = i & ((1u << vpr_log2) - 1u);
            const uint32_t row = i >> vpr_log2;  // s * H + h of the destination
            const uint32_t s = row / H, h = row - s * H;
            const uint32_t g = h / Hp, j = h - g * Hp;
            const uint32_t src = (((g * S + s) * Hp + j) << vpr_log2) + part;
            ok[u] = in_bounds(st, src, 1, total, kTagHead2Seq, 1);
            if (ok[u]) v[u] = __ldcs(in + src);
        }
    }
#pragma unroll
    for (int u = 0; u < kLayoutUnroll; ++u) {
        if (ok[u]) __stcs(out + base + u * kLayoutThreads, v[u]);
    }
}

// head2seq for a chunk of one group's heads: group g's buffer [S][H/P][D],
// heads [j0, j0 + jc) -> out[s][g*(H/P) + j].  Used to overlap the output
// exchange of one head chunk with the attention of the next.
__global__ void __launch_bounds__(kLayoutThreads) head2seq_heads_kernel(const uint4* __restrict__ in,
                                                                        uint4* __restrict__ out, uint32_t H,
                                                                        uint32_t Hp, uint32_t hbase, uint32_t j0,
                                                                        uint32_t jc, uint32_t vpr_log2,
                                                                        uint32_t total, uint32_t in_extent,
                                                                        uint32_t out_extent, DeviceStatus* st) {
    const uint32_t base = blockIdx.x * (kLayoutThreads * kLayoutUnroll) + threadIdx.x;
    uint4 v[kLayoutUnroll];
    bool ok[kLayoutUnroll];
#pragma unroll
    for (int u = 0; u < kLayoutUnroll; ++u) {
        const uint32_t i = base + u * kLayoutThreads;
        ok[u] = false;
        if (i < total) {
            const uint32_t part = i & ((1u << vpr_log2) - 1u);
            const uint32_t rest = i >> vpr_log2;  // s * jc + jj
            const uint32_t s = rest / jc, jj = rest - s * jc;
            const uint32_t src = ((s * Hp + j0 + jj) << vpr_log2) + part;
            ok[u] = in_bounds(st, src, 1, in_extent, kTagHead2SeqHeads, 1);
            if (ok[u]) v[u] = __ldcs(in + src);
        }
    }
#pragma unroll
    for (int u = 0; u < kLayoutUnroll; ++u) {
        const uint32_t i = base + u * kLayoutThreads;
        if (ok[u]) {
            const uint32_t part = i & ((1u << vpr_log2) - 1u);
            const uint32_t rest = i >> vpr_log2;
            const uint32_t s = rest / jc, jj = rest - s * jc;
            const uint32_t dst = ((s * H + hbase + j0 + jj) << vpr_log2) + part;
            if (in_bounds(st, dst, 1, out_extent, kTagHead2SeqHeads, 2)) __stcs(out + dst, v[u]);
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
    const uint32_t in_extent = static_cast<uint32_t>(static_cast<uint64_t>(S) * Hp << vpr_log2);
    const uint32_t out_extent = static_cast<uint32_t>(static_cast<uint64_t>(S) * H << vpr_log2);
    DeviceStatus* st = nullptr;
    const int rc = device_status_ptr(&st);
    if (rc != H3ATTN_OK) return rc;
    head2seq_heads_kernel<<<(total + per_block - 1) / per_block, kLayoutThreads, 0, stream>>>(
        static_cast<const uint4*>(in_group), static_cast<uint4*>(out), H, Hp, g * Hp, j0, jc, vpr_log2, total,
        in_extent, out_extent, st);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? H3ATTN_OK : cuda_fail(e);
}

// `out_short`: vectors by which the output extent given to seq2head is
// understated (0, except in the bounds self-test).
static int launch_layout(bool to_heads, const void* in, void* out, int S, int H, int D, int P, cudaStream_t stream,
                         uint32_t out_short = 0) {
    const uint32_t vpr_log2 = (D == 128) ? 4u : 3u;  // 16-byte vectors per head row
    const uint64_t total64 = static_cast<uint64_t>(S) * H * (static_cast<uint64_t>(D) / 8);
    if (total64 == 0) return H3ATTN_OK;
    const uint32_t total = static_cast<uint32_t>(total64);
    const uint32_t per_block = kLayoutThreads * kLayoutUnroll;
    const uint32_t blocks = (total + per_block - 1) / per_block;
    DeviceStatus* st = nullptr;
    const int rc = device_status_ptr(&st);
    if (rc != H3ATTN_OK) return rc;
    if (to_heads)
        seq2head_kernel<<<blocks, kLayoutThreads, 0, stream>>>(static_cast<const uint4*>(in), static_cast<uint4*>(out),
                                                               S, H, H / P, vpr_log2, total, total - out_short, st);
    else
        head2seq_kernel<<<blocks, kLayoutThreads, 0, stream>>>(static_cast<const uint4*>(in), static_cast<uint4*>(out),
                                                               S, H, H / P, vpr_log2, total, st);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? H3ATTN_OK : cuda_fail(e);
}

int launch_seq2head(const void* in, void* out, int S, int H, int D, int P, cudaStream_t stream) {
    return launch_layout(true, in, out, S, H, D, P, stream);
}

int launch_head2seq(const void* in, void* out, int S, int H, int D, int P, cudaStream_t stream) {
    return launch_layout(false, in, out, S, H, D, P, stream);
}

// Bounds self-test: seq2head of S = 2, H = 2, D = 64, P = 2 (32 vectors in,
// 32 out) from buf[0, 512) to buf[512, 1024), told that the output holds 31
// vectors.  Exactly one store (output vector 31, which does exist) fails the
// check.
int launch_selftest_bounds(void* buf, cudaStream_t stream) {
    uint8_t* b = static_cast<uint8_t*>(buf);
    return launch_layout(true, b, b + 512, 2, 2, 64, 2, stream, 1);
}

}  // namespace h3
