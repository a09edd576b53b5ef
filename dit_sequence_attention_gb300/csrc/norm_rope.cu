// norm_rope.cu -- fused QK-RMSNorm + three-axis rotary embedding.
//
// "[feat] Tensor parallelism for MiniMax-H3" (diffusers PR #14609), PR
// description: QK-norms are head_dim-shaped and applied after the head split;
// the rotary embedding uses real sin/cos, broadcasts over heads, and its angle
// is inv_freq times the position.  Per (token, head) row of q and of k:
//     y = x / sqrt(mean(x^2) + eps) * w;   pair i of axis a rotated by pos_a * theta^(-2i/d_a).
//
// One block of 128 threads per token.  The token's D/2 rotation angles are shared by all
// 2*H rows (q and k, every head), so the block computes cos/sin once: the
// angle pos * inv_freq and its reduction to [-pi, pi] in fp64 (a handful of
// fp64 ops per pair; the position is an exact integer, so the reduced angle
// is accurate to ~1e-16 even for positions in the thousands), then sincosf on
// the reduced fp32 angle.  Each thread owns 8 consecutive dims (one 16-byte
// vector) of a row, i.e. 4 whole rotation pairs; the D/8 threads of a row
// reduce the sum of squares with warp shuffles.  A thread sits at the same
// place in every row it handles, so it folds its 8 weights into its 4 pairs'
// rotations once per token (out = inv * (f0 * w0 * (c, s) + f1 * w1 * (-s, c)),
// three packed f32x2 operations per pair) and q and k are done one after the
// other, each with its own folded coefficients.  Loads are issued four
// vectors per thread at a time, the first batch before the angle work;
// results leave with streaming (evict-first) stores.  Small blocks (64
// registers a thread) keep 8 tokens in flight per SM.
// HBM-bound: 4 * H * D * 2 bytes per token (read and write q and k).
//
// With P > 1 the results are written straight into the Ulysses head-sharded
// layout [P][S][H/P][D] (the layout seq2head produces), so the normalised q
// and k never make a token-major round trip through HBM before the exchange.
// That store is a separate instantiation (kSharded) and finds a head's group
// by a multiply-shift reciprocal of H/P instead of an integer division per
// vector (the division alone cost 14 % of the kernel's time).
#include <cmath>
#include <cstdint>

#include "h3_device.cuh"
#include "h3_internal.h"

namespace h3 {

constexpr int kNormThreads = 128;
constexpr int kNormMaxVec = 4;  // vectors per thread held in registers per pass

struct RopeTable {
    double inv_freq[64];   // per rotation pair p = (global dim)/2
    int axis[64];          // 0 = t, 1 = h, 2 = w
};

// kSharded: write the head-sharded layout [P][S][H/P][D] (one batch item)
// instead of the input's token-major one.
template <int D, bool kSharded>
__global__ void __launch_bounds__(kNormThreads) norm_rope_kernel(
    const uint4* q, const uint4* k, uint4* qo, uint4* ko, float* __restrict__ dbg,
    const float* __restrict__ wq, const float* __restrict__ wk, const int32_t* __restrict__ pos, int S, int H,
    float eps, size_t dbg_k_offset, int P, const RopeTable tab, size_t n_vec, DeviceStatus* st, int Hp,
    unsigned long long hp_recip) {
    // n_vec: 16-byte vectors in each of q, k, q_out, k_out (B * S * H * D / 8);
    // st: device status word (debug-check builds).
    constexpr int VPR = D / 8;  // vectors per row
    constexpr double kTwoPi = 6.283185307179586476925286766559;
    constexpr double kInvTwoPi = 0.15915494309189533576888376337251;
    __shared__ float2 cs[D / 2];

    const int tok = blockIdx.x;  // b * S + s
    const int s = tok % S;
    const int cpt = H * VPR;      // vectors per tensor for this token
    const size_t tok_vec = static_cast<size_t>(tok) * cpt;
    const float inv_d = 1.0f / static_cast<float>(D);

    // This thread's position in a row, part = (vector index) % VPR, is the same
    // for every vector it handles (the block size is a multiple of VPR and so is
    // the tensor's vector count per token), so its 4 rotation pairs and 8
    // weights are loaded once per token.
    const int part = static_cast<int>(threadIdx.x) % VPR;

    // Issue the first batch of q loads before anything else, so their latency
    // overlaps the position load and the angle computation below.
    const int iters = (cpt + kNormThreads - 1) / kNormThreads;  // per tensor
    uint4 x[kNormMaxVec];
#pragma unroll
    for (int u = 0; u < kNormMaxVec; ++u) {
        const int idx = u * kNormThreads + threadIdx.x;
        x[u] = make_uint4(0, 0, 0, 0);
        if (u < iters && idx < cpt && in_bounds(st, tok_vec + idx, 1, n_vec, kTagNormRope, 1))
            x[u] = __ldcs(q + tok_vec + idx);
    }
    if (threadIdx.x < D / 2) {
        const int pr = threadIdx.x;
        const int pidx = 3 * s + tab.axis[pr];
        const int32_t pv = in_bounds(st, pidx, 1, 3ull * S, kTagNormRope, 2) ? __ldg(pos + pidx) : 0;
        const double ang = static_cast<double>(pv) * tab.inv_freq[pr];
        const double turns = rint(ang * kInvTwoPi);
        const float red = static_cast<float>(fma(-turns, kTwoPi, ang));
        float sn, c;
        sincosf(red, &sn, &c);
        cs[pr] = make_float2(c, sn);
    }
    __syncthreads();
    float2 rot[4];
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) rot[pp] = cs[part * 4 + pp];

#pragma unroll 1
    for (int t = 0; t < 2; ++t) {  // q, then k
        const uint4* src = t ? k : q;
        uint4* out = t ? ko : qo;
        // weight and rotation folded per pair (y0, y1) of this thread's 8 dims:
        //   out0 = inv * (f0 * w0 c - f1 * w1 s),  out1 = inv * (f0 * w0 s + f1 * w1 c)
        uint64_t ca[4], cb[4];
        {
            const float* w = (t ? wk : wq) + part * 8;
            float wv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (in_bounds(st, static_cast<size_t>(part) * 8, 8, D, kTagNormRope, 4)) {
                const float4 wa = __ldg(reinterpret_cast<const float4*>(w));
                const float4 wb = __ldg(reinterpret_cast<const float4*>(w) + 1);
                wv[0] = wa.x; wv[1] = wa.y; wv[2] = wa.z; wv[3] = wa.w;
                wv[4] = wb.x; wv[5] = wb.y; wv[6] = wb.z; wv[7] = wb.w;
            }
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
                const float w0 = wv[2 * pp], w1 = wv[2 * pp + 1], c = rot[pp].x, sn = rot[pp].y;
                ca[pp] = f2_pack(w0 * c, w0 * sn);
                cb[pp] = f2_pack(-(w1 * sn), w1 * c);
            }
        }
        for (int it0 = 0; it0 < iters; it0 += kNormMaxVec) {
            if (it0 > 0 || t > 0) {
#pragma unroll
                for (int u = 0; u < kNormMaxVec; ++u) {
                    const int idx = (it0 + u) * kNormThreads + threadIdx.x;
                    x[u] = make_uint4(0, 0, 0, 0);
                    if (it0 + u < iters && idx < cpt && in_bounds(st, tok_vec + idx, 1, n_vec, kTagNormRope, 3))
                        x[u] = __ldcs(src + tok_vec + idx);
                }
            }
#pragma unroll
            for (int u = 0; u < kNormMaxVec; ++u) {
                if (it0 + u >= iters) break;  // uniform across the block
                const int c = (it0 + u) * kNormThreads + threadIdx.x;  // vector index within the token's tensor
                const uint32_t w4[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
                float f[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    f[2 * e] = bf16lo_to_f32(w4[e]);
                    f[2 * e + 1] = bf16hi_to_f32(w4[e]);
                }
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
#pragma unroll
                for (int off = VPR / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                if (c >= cpt) continue;
                const float inv = rsqrtf(ss * inv_d + eps);
                const uint64_t inv2 = f2_pack(inv, inv);
                float y[8];
#pragma unroll
                for (int pp = 0; pp < 4; ++pp) {
                    const uint64_t r = f2_mul(f2_fma(f2_pack(f[2 * pp + 1], f[2 * pp + 1]), cb[pp],
                                                     f2_mul(f2_pack(f[2 * pp], f[2 * pp]), ca[pp])),
                                              inv2);
                    f2_unpack(r, y[2 * pp], y[2 * pp + 1]);
                }
                uint4 o;
                o.x = pack_bf16x2(y[0], y[1]);
                o.y = pack_bf16x2(y[2], y[3]);
                o.z = pack_bf16x2(y[4], y[5]);
                o.w = pack_bf16x2(y[6], y[7]);
                size_t dst = tok_vec + c;
                if (kSharded) {  // head-sharded output: [g][s][j] with h = g * (H/P) + j
                    const int h = c / VPR;
                    // g = h / Hp by multiply and shift (hp_recip = ceil(2^32 / Hp); exact for h < 2^16)
                    const int g = static_cast<int>((static_cast<unsigned long long>(h) * hp_recip) >> 32);
                    dst = ((static_cast<size_t>(g) * S + s) * Hp + (h - g * Hp)) * VPR + part;
                }
                if (in_bounds(st, dst, 1, n_vec, kTagNormRope, 5)) __stcs(out + dst, o);
                if (dbg != nullptr &&
                    in_bounds(st, (t ? dbg_k_offset : 0) + (tok_vec + c) * 8, 8, 2 * dbg_k_offset, kTagNormRope, 6)) {
                    float4* d4 = reinterpret_cast<float4*>(dbg + (t ? dbg_k_offset : 0) + (tok_vec + c) * 8);
                    d4[0] = make_float4(y[0], y[1], y[2], y[3]);
                    d4[1] = make_float4(y[4], y[5], y[6], y[7]);
                }
            }
        }
    }
}

int launch_norm_rope(const void* q, const void* k, void* q_out, void* k_out, float* dbg, const float* w_q,
                     const float* w_k, const int32_t* pos, int B, int S, int H, int D, int d_t, int d_h, int d_w,
                     float eps, double theta, int P, cudaStream_t stream) {
    RopeTable tab;
    const int width[3] = {d_t, d_h, d_w};
    int pr = 0;
    for (int a = 0; a < 3; ++a) {
        for (int i = 0; i < width[a] / 2; ++i, ++pr) {
            tab.inv_freq[pr] = std::pow(theta, -2.0 * static_cast<double>(i) / static_cast<double>(width[a]));
            tab.axis[pr] = a;
        }
    }
    for (; pr < 64; ++pr) {
        tab.inv_freq[pr] = 0.0;
        tab.axis[pr] = 0;
    }
    const size_t dbg_k = static_cast<size_t>(B) * S * H * D;
    const size_t n_vec = dbg_k / 8;
    const unsigned blocks = static_cast<unsigned>(B) * static_cast<unsigned>(S);
    if (blocks == 0) return H3ATTN_OK;
    DeviceStatus* st = nullptr;
    const int rc = device_status_ptr(&st);
    if (rc != H3ATTN_OK) return rc;
    const int Hp = H / P;
    const unsigned long long hp_recip = ((1ull << 32) + static_cast<unsigned long long>(Hp) - 1) / Hp;
    auto launch = [&](auto kernel) {
        kernel<<<blocks, kNormThreads, 0, stream>>>(
            static_cast<const uint4*>(q), static_cast<const uint4*>(k), static_cast<uint4*>(q_out),
            static_cast<uint4*>(k_out), dbg, w_q, w_k, pos, S, H, eps, dbg_k, P, tab, n_vec, st, Hp, hp_recip);
    };
    if (D == 128) {
        if (P > 1) launch(norm_rope_kernel<128, true>);
        else launch(norm_rope_kernel<128, false>);
    } else {
        if (P > 1) launch(norm_rope_kernel<64, true>);
        else launch(norm_rope_kernel<64, false>);
    }
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? H3ATTN_OK : cuda_fail(e);
}

}  // namespace h3
