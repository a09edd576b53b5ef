// attention.cu -- exact masked multi-head attention on sm_103a tensor cores.
//
// What it computes ("buqi-minimax-h3-multigpu" README, "On accuracy" / "How
// it works": exact full attention over the whole packed sequence for a subset
// of heads; padded keys beyond kv_len carry no weight):
//     o[i] = sum_{j < kv_len} softmax_j(scale * q[i].k[j]) v[j]      per head.
//
// How (one CTA = one head x 256 query rows, 320 threads):
//   warp 8      TMA producer: Q tiles once, then K/V tiles of 128 keys into a
//               three-stage key ring and a two-stage value ring (128B-swizzled
//               boxes of 64 columns).
//   warp 9      allocates 512 TMEM columns, one lane issues every tcgen05.mma:
//               S_i = Q_i K^T (both operands in shared memory) and
//               O_i += P_i V   (P from TMEM, V from shared memory, MN-major).
//               A thread that waits on an mbarrier lets the MMAs it has queued
//               drain, so its only waits between MMA groups are those for P;
//               the TMA barriers of a step are waited after the last group of
//               the step before.
//   warps 0-3   softmax for query tile 0 (rows 0..127), warps 4-7 for tile 1.
//               Thread = one query row = one TMEM lane: the 128 scores arrive in
//               one 128-column TMEM load; row max with three-input max; then the
//               exp2 arguments for the whole row (packed f32x2 FMA), all 128
//               exponentials, and the packed sums and bf16 pairs -- phase-ordered
//               so the exponentials run back to back on the MUFU pipe while the
//               other pipes work; P is written back over S as bf16 pairs; O is
//               rescaled in TMEM only when the running max grows by more than
//               2^8 (otherwise the stale max is kept, which is exact after the
//               final division).
// The two query tiles ping-pong: while one tile's softmax runs, the tensor
// core works on the other tile's products.  The key tail is masked by giving
// the K/V tensor maps an extent of kv_len (TMA fills zeros, never reads pad
// rows) and by setting scores of keys >= kv_len to -inf.  The per-row
// reduction order depends only on kv_len, never on the head range or grid,
// so any split of the heads over calls is bit-identical.
#include <cuda.h>

#include "h3_device.cuh"
#include "h3_internal.h"

namespace h3 {

constexpr int kAttnThreads = 320;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8

#ifndef H3_ATTN_KSTAGES
#define H3_ATTN_KSTAGES 3
#endif
#ifndef H3_ATTN_VSTAGES
#define H3_ATTN_VSTAGES 2
#endif

template <int D>
struct AttnTraits {
    static constexpr int BM = 128;                       // query rows per tile (TMEM lanes)
    static constexpr int BN = 128;                       // keys per tile
    static constexpr int KST = H3_ATTN_KSTAGES;          // key ring depth
    static constexpr int VST = H3_ATTN_VSTAGES;          // value ring depth
    static constexpr int NCHUNK = D / 64;                // 128-byte swizzle boxes along head_dim
    static constexpr int CHUNK_BYTES = 128 * 128;        // 128 rows x 64 bf16
    static constexpr int TILE_BYTES = NCHUNK * CHUNK_BYTES;
    static constexpr int OFF_Q = 0;                      // 2 query tiles
    static constexpr int OFF_K = 2 * TILE_BYTES;         // KST key stages
    static constexpr int OFF_V = OFF_K + KST * TILE_BYTES;  // VST value stages
    static constexpr int OFF_BAR = OFF_V + VST * TILE_BYTES;
    static constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;  // barriers + 1 KB alignment slack
    static_assert(KST >= 2 && KST <= 4 && VST >= 2 && VST <= 4, "ring depth");
    static_assert(SMEM_BYTES <= 232448, "shared memory per block");
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 256 + D;
    static constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, false, false);
    static constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, D, false, true);
};

// Barrier slots (8 bytes each) in the barrier area (room for up to 4 stages per ring).
enum : int {
    B_QFULL = 0,
    B_KFULL = 1,    // +stage
    B_VFULL = 5,    // +stage
    B_KEMPTY = 9,   // +stage
    B_VEMPTY = 13,  // +stage
    B_SFULL = 17,   // +query tile
    B_PFULL = 19,   // +query tile
    B_OFINAL = 21,  // +query tile
    B_DRAIN = 23,
    B_COUNT = 24
};

struct AttnParams {
    __nv_bfloat16* o;   // this batch item's output [S][H_buf][D]
    int S;
    int H_buf;
    int head_begin;
    int kv_len;
    int n_kv_tiles;
    float scale_log2;   // softmax scale * log2(e)
    unsigned long long wait_limit_ns;
    DeviceStatus* status;
    unsigned long long o_elems;  // S * H_buf * D: extent of `o` (index checks of debug-check builds)
};

// Wait for an mbarrier phase ignoring the abort flag (used only on the abort
// path to let copies already in flight land before the CTA exits).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) break;
    }
}

// Issue S = Q K^T: eight K=16 steps.  The descriptors are built once per CTA;
// each step only adds a compile-time offset to the start-address field, so
// the single issuing thread keeps up with the tensor core (rebuilding a
// descriptor per instruction costs more than the 64-cycle MMA itself).
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t dq, uint64_t dk) {
    using T = AttnTraits<D>;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = static_cast<uint64_t>(((kk / 4) * T::CHUNK_BYTES + (kk % 4) * 32) >> 4);
        mma_ss(d_tmem, dq + off, dk + off, T::IDESC_QK, kk > 0 ? 1u : 0u);
    }
}

// Issue O (+)= P V: eight K=16 steps over the tile's 128 keys.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t dv, bool accumulate) {
    using T = AttnTraits<D>;
#pragma unroll
    for (int kk = 0; kk < T::BN / 16; ++kk) {
        // 16 keys per instruction: P columns (bf16 pairs) [8kk, 8kk+8), V rows [16kk, 16kk+16).
        mma_ts(d_tmem, p_tmem + kk * 8, dv + static_cast<uint64_t>((kk * 2048) >> 4), T::IDESC_PV,
               (accumulate || kk > 0) ? 1u : 0u);
    }
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    using T = AttnTraits<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - raw);
    const uint32_t bar0 = sbase + T::OFF_BAR;
    auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + T::OFF_BAR + 8 * B_COUNT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + T::OFF_BAR + 8 * B_COUNT + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int head = p.head_begin + static_cast<int>(blockIdx.y);
    const int q0 = static_cast<int>(blockIdx.x) * 2 * T::BM;
    const int n = p.n_kv_tiles;

    if (threadIdx.x == 0) {
        mbar_init(bar(B_QFULL), 1);
        for (int s = 0; s < T::KST; ++s) {
            mbar_init(bar(B_KFULL + s), 1);
            mbar_init(bar(B_KEMPTY + s), 1);
        }
        for (int s = 0; s < T::VST; ++s) {
            mbar_init(bar(B_VFULL + s), 1);
            mbar_init(bar(B_VEMPTY + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(B_SFULL + t), 1);
            mbar_init(bar(B_PFULL + t), 4);   // one elected lane per softmax warp
            mbar_init(bar(B_OFINAL + t), 1);
        }
        mbar_init(bar(B_DRAIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 9) {
        tmem_alloc<512>(smem_u32(tmem_slot));
        tmem_relinquish();
    }
    if (warp == 8 && lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl ctl{abort_flag, p.wait_limit_ns, p.status, kTagAttention};

    const uint32_t sQ = sbase + T::OFF_Q, sK = sbase + T::OFF_K, sV = sbase + T::OFF_V;

    if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t keep = l2_policy_evict_last();   // K/V: reused by every query block of the head
            const uint64_t once = l2_policy_evict_first();  // Q: read once
            int last_k = -1, last_v = -1;                   // last tile index issued per ring
            mbar_arrive_expect_tx(bar(B_QFULL), 2 * T::TILE_BYTES);
            for (int t = 0; t < 2; ++t)
                for (int c = 0; c < T::NCHUNK; ++c)
                    tma_load_3d_hint(sQ + t * T::TILE_BYTES + c * T::CHUNK_BYTES, &tmQ, bar(B_QFULL), c * 64,
                                     head, q0 + t * T::BM, once);
            for (int j = 0; j < n; ++j) {
                const int ks = j % T::KST, ku = j / T::KST;
                if (ku > 0 && !mbar_wait(bar(B_KEMPTY + ks), (ku - 1) & 1, ctl, 1)) break;
                mbar_arrive_expect_tx(bar(B_KFULL + ks), T::TILE_BYTES);
                for (int c = 0; c < T::NCHUNK; ++c)
                    tma_load_3d_hint(sK + ks * T::TILE_BYTES + c * T::CHUNK_BYTES, &tmK, bar(B_KFULL + ks), c * 64,
                                     head, j * T::BN, keep);
                last_k = j;
                const int vs = j % T::VST, vu = j / T::VST;
                if (vu > 0 && !mbar_wait(bar(B_VEMPTY + vs), (vu - 1) & 1, ctl, 2)) break;
                mbar_arrive_expect_tx(bar(B_VFULL + vs), T::TILE_BYTES);
                for (int c = 0; c < T::NCHUNK; ++c)
                    tma_load_3d_hint(sV + vs * T::TILE_BYTES + c * T::CHUNK_BYTES, &tmV, bar(B_VFULL + vs), c * 64,
                                     head, j * T::BN, keep);
                last_v = j;
            }
            if (*abort_flag) {  // let every copy already issued land before the CTA exits
                const uint64_t lim = p.wait_limit_ns;
                drain_wait(bar(B_QFULL), 0, lim);
                for (int j = last_k; j >= 0 && j > last_k - T::KST; --j)
                    drain_wait(bar(B_KFULL + j % T::KST), (j / T::KST) & 1, lim);
                for (int j = last_v; j >= 0 && j > last_v - T::VST; --j)
                    drain_wait(bar(B_VFULL + j % T::VST), (j / T::VST) & 1, lim);
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint64_t dQ0 = smem_desc_sw128(sQ, 16, 1024);
            const uint64_t dQ1 = smem_desc_sw128(sQ + T::TILE_BYTES, 16, 1024);
            const uint64_t dK = smem_desc_sw128(sK, 16, 1024);               // + stage * TILE_BYTES / 16
            const uint64_t dV = smem_desc_sw128(sV, T::CHUNK_BYTES, 1024);   // + stage * TILE_BYTES / 16
            constexpr uint64_t kStage = T::TILE_BYTES >> 4;
            bool ok = mbar_wait(bar(B_QFULL), 0, ctl, 10) && mbar_wait(bar(B_KFULL + 0), 0, ctl, 11);
            if (ok) {
                tc_fence_after_sync();
                issue_qk<D>(tmem + T::COL_S0, dQ0, dK);
                mma_commit(bar(B_SFULL + 0));
                issue_qk<D>(tmem + T::COL_S1, dQ1, dK);
                mma_commit(bar(B_SFULL + 1));
                mma_commit(bar(B_KEMPTY + 0));
            }
            // The TMA barriers of the next step are waited right after the last
            // MMA group of this one, where the thread would soon wait for P
            // anyway: a waiting thread lets its queued MMAs drain, so between
            // PV_0 and QK_0 (and PV_1, QK_1) the stream is never broken.
            ok = ok && mbar_wait(bar(B_VFULL + 0), 0, ctl, 12) && (n < 2 || mbar_wait(bar(B_KFULL + 1 % T::KST), 0, ctl, 14));
            for (int j = 0; j < n && ok; ++j) {
                const int vs = j % T::VST;
                const bool more = (j + 1) < n;
                const int ks = (j + 1) % T::KST;
                const uint64_t dVj = dV + vs * kStage;
                if (!mbar_wait(bar(B_PFULL + 0), j & 1, ctl, 13)) { ok = false; break; }
                tc_fence_after_sync();
                issue_pv<D>(tmem + T::COL_O0, tmem + T::COL_S0, dVj, j > 0);
                if (more) {
                    issue_qk<D>(tmem + T::COL_S0, dQ0, dK + ks * kStage);
                    mma_commit(bar(B_SFULL + 0));
                } else {
                    mma_commit(bar(B_OFINAL + 0));
                }
                if (!mbar_wait(bar(B_PFULL + 1), j & 1, ctl, 15)) { ok = false; break; }
                tc_fence_after_sync();
                issue_pv<D>(tmem + T::COL_O1, tmem + T::COL_S1, dVj, j > 0);
                mma_commit(bar(B_VEMPTY + vs));
                if (more) {
                    issue_qk<D>(tmem + T::COL_S1, dQ1, dK + ks * kStage);
                    mma_commit(bar(B_SFULL + 1));
                    mma_commit(bar(B_KEMPTY + ks));
                    // next step's V tile and the key tile after next
                    const int jv = j + 1, jk = j + 2;
                    if (!mbar_wait(bar(B_VFULL + jv % T::VST), (jv / T::VST) & 1, ctl, 12) ||
                        (jk < n && !mbar_wait(bar(B_KFULL + jk % T::KST), (jk / T::KST) & 1, ctl, 14))) {
                        ok = false;
                        break;
                    }
                } else {
                    mma_commit(bar(B_OFINAL + 1));
                }
            }
            if (!ok) {  // no tensor-core work may still be running when TMEM is freed
                mma_commit(bar(B_DRAIN));
                drain_wait(bar(B_DRAIN), 0, p.wait_limit_ns);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int wg = warp >> 2;          // query tile
        const int wq = warp & 3;           // TMEM lane quarter
        const int row_in_tile = wq * 32 + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const uint32_t colS = wg ? T::COL_S1 : T::COL_S0;
        const uint32_t colO = wg ? T::COL_O1 : T::COL_O0;
        const float sl2 = p.scale_log2;
        const int tail = p.kv_len - (n - 1) * T::BN;  // valid keys in the last tile, 1..128
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            // warp-uniform outcome: the TMEM accessors below are warp-collective
            if (!__all_sync(0xffffffffu, mbar_wait(bar(B_SFULL + wg), j & 1, ctl, 20 + wg))) { ok = false; break; }
            tc_fence_after_sync();
            float s[T::BN];
            tmem_ld128(lane_addr + colS, s);
            if (j == n - 1 && tail < T::BN) {
#pragma unroll
                for (int c = 0; c < T::BN; ++c)
                    if (c >= tail) s[c] = -INFINITY;
            }
            // row max: eight independent chains of three-input max, then a tree
            float mx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
            for (int c = 16; c < T::BN; c += 16) {
#pragma unroll
                for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], s[c + 2 * i], s[c + 2 * i + 1]);
            }
            const float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * sl2;
            const bool need = (j > 0) && (mt > m + kRescaleThreshold);
            if (__any_sync(0xffffffffu, need)) {
                const float alpha = need ? ex2_approx(m - mt) : 1.0f;
                const uint64_t alpha2 = f2_pack(alpha, alpha);
#pragma unroll
                for (int c = 0; c < D / 16; ++c) {
                    float o16[16];
                    uint32_t w16[16];
                    tmem_ld16(lane_addr + colO + 16 * c, o16);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float a, b;
                        f2_unpack(f2_mul(f2_pack(o16[2 * i], o16[2 * i + 1]), alpha2), a, b);
                        w16[2 * i] = __float_as_uint(a);
                        w16[2 * i + 1] = __float_as_uint(b);
                    }
                    tmem_st16(lane_addr + colO + 16 * c, w16);
                }
                tmem_wait_st();
                l *= alpha;
            }
            if (j == 0 || need) m = mt;
            // p = exp2(s * scale*log2e - m): the argument as packed fp32 pairs, the
            // sums in four packed accumulators; P (bf16 pairs) overwrites the first
            // BN/2 columns of S, 32 keys at a time (stores complete at the wait below).
            const uint64_t sl2x2 = f2_pack(sl2, sl2);
            const uint64_t negm2 = f2_pack(-m, -m);
            // arguments for all 128 keys, then all exponentials, then sums and packs
#pragma unroll
            for (int i = 0; i < T::BN / 2; ++i) {
                float a0, a1;
                f2_unpack(f2_fma(f2_pack(s[2 * i], s[2 * i + 1]), sl2x2, negm2), a0, a1);
                s[2 * i] = a0;
                s[2 * i + 1] = a1;
            }
#pragma unroll
            for (int i = 0; i < T::BN; ++i) s[i] = ex2_approx(s[i]);
            uint64_t acc[8] = {0ull, 0ull, 0ull, 0ull, 0ull, 0ull, 0ull, 0ull};
#pragma unroll
            for (int c = 0; c < T::BN / 32; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float p0 = s[32 * c + 2 * i], p1 = s[32 * c + 2 * i + 1];
                    acc[i & 7] = f2_add(acc[i & 7], f2_pack(p0, p1));
                    pk[i] = pack_bf16x2(p0, p1);
                }
                tmem_st16(lane_addr + colS + 16 * c, pk);
            }
            {
                float a0, a1;
                f2_unpack(f2_add(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])),
                                 f2_add(f2_add(acc[4], acc[5]), f2_add(acc[6], acc[7]))), a0, a1);
                l += a0 + a1;
            }
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_PFULL + wg));
        }
        // ---------------------------------------------------------- epilogue
        if (ok && __all_sync(0xffffffffu, mbar_wait(bar(B_OFINAL + wg), 0, ctl, 24 + wg))) {
            tc_fence_after_sync();
            const float inv_l = 1.0f / l;
            const int row = q0 + wg * T::BM + row_in_tile;
            __nv_bfloat16* dst = p.o + (static_cast<size_t>(row) * p.H_buf + head) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float o32[32];
                tmem_ld32(lane_addr + colO + 32 * c, o32);
                if (row < p.S && in_bounds(p.status, (static_cast<size_t>(row) * p.H_buf + head) * D + 32 * c, 32,
                                           p.o_elems, kTagAttention, 1)) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 w;
                        w.x = pack_bf16x2(o32[8 * v + 0] * inv_l, o32[8 * v + 1] * inv_l);
                        w.y = pack_bf16x2(o32[8 * v + 2] * inv_l, o32[8 * v + 3] * inv_l);
                        w.z = pack_bf16x2(o32[8 * v + 4] * inv_l, o32[8 * v + 5] * inv_l);
                        w.w = pack_bf16x2(o32[8 * v + 6] * inv_l, o32[8 * v + 7] * inv_l);
                        d4[v] = w;
                    }
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after_sync();
        tmem_dealloc<512>(tmem);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static int encode_rows_map(CUtensorMap* m, const void* base, int D, int H_buf, int rows) {
    // dims innermost first: head_dim, head, sequence row; box = 64 x 1 x 128.
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H_buf),
                                static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H_buf) * D * 2};
    const cuuint32_t box[3] = {64, 1, 128};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                             CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int D>
static int launch_one(const void* q, const void* k, const void* v, void* o, int S, int H_buf, int head_begin,
                      int head_count, int kv_len, float scale, cudaStream_t stream) {
    using T = AttnTraits<D>;
    int rc = ensure_smem_attr(reinterpret_cast<const void*>(attn_fwd_kernel<D>), T::SMEM_BYTES);
    if (rc != H3ATTN_OK) return rc;
    CUtensorMap mq, mk, mv;
    if ((rc = encode_rows_map(&mq, q, D, H_buf, S)) != H3ATTN_OK) return rc;
    if ((rc = encode_rows_map(&mk, k, D, H_buf, kv_len)) != H3ATTN_OK) return rc;
    if ((rc = encode_rows_map(&mv, v, D, H_buf, kv_len)) != H3ATTN_OK) return rc;
    AttnParams prm;
    prm.o = static_cast<__nv_bfloat16*>(o);
    prm.S = S;
    prm.H_buf = H_buf;
    prm.head_begin = head_begin;
    prm.kv_len = kv_len;
    prm.n_kv_tiles = (kv_len + T::BN - 1) / T::BN;
    prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    prm.wait_limit_ns = wait_limit_ns();
    prm.o_elems = static_cast<unsigned long long>(S) * H_buf * D;
    if ((rc = device_status_ptr(&prm.status)) != H3ATTN_OK) return rc;
    const dim3 grid(static_cast<unsigned>((S + 2 * T::BM - 1) / (2 * T::BM)), static_cast<unsigned>(head_count));
    attn_fwd_kernel<D><<<grid, kAttnThreads, T::SMEM_BYTES, stream>>>(mq, mk, mv, prm);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? H3ATTN_OK : cuda_fail(e);
}

int launch_attention(const void* q, const void* k, const void* v, void* o, int S, int H_buf, int D, int head_begin,
                     int head_count, int kv_len, float scale, cudaStream_t stream) {
    if (D == 128) return launch_one<128>(q, k, v, o, S, H_buf, head_begin, head_count, kv_len, scale, stream);
    return launch_one<64>(q, k, v, o, S, H_buf, head_begin, head_count, kv_len, scale, stream);
}

}  // namespace h3
