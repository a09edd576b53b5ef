// qkv_proj.cu -- the all-gather exchange variant's QKV projection on sm_103a
// tensor cores (FP8 E4M3 x E4M3 -> fp32, tcgen05.mma kind::f8f6f4).
//
// "buqi-minimax-h3-multigpu" README, "How it works": for world sizes up to 4
// every rank receives the whole modulated hidden state and multiplies it by
// only its own head rows of qkv_proj; slicing the fp8 weight by rows is exact
// because its scale is one number per tensor.  For rank r of P:
//     out_part[s][c] = scale * sum_e x[s][e] * w[part*inner + r*inner/P + c][e]
// for part in (q, k, v) and c < inner/P, written as bf16 [S][inner/P] per part
// (the head-sharded [S][H/P][D] layout the attention kernel reads).
//
// Persistent: one CTA per SM walks output tiles of 128 tokens x 256 output
// features of one part (tile t, t + grid, ...), 192 threads:
//   warp 0      TMA producer: x and w slices of 128 bytes along K into a
//               4-stage ring (128B swizzle) that runs across tiles.
//   warp 1      allocates 512 TMEM columns = two 128x256 fp32 accumulators;
//               one lane issues 4 MMAs (K = 32) per stage with descriptors
//               built once (start-address offsets only).
//   warps 2-5   epilogue: TMEM -> registers, times scale, bf16, global stores;
//               while they drain one accumulator the MMAs fill the other.
// Every CTA loads its own operands, with plain TMA copies into its own shared memory.
// Tiles are numbered with the output-feature tile fastest, so the CTAs that
// run at the same time share their x rows through L2; the weight slice
// (58 MB at P = 2) stays L2-resident.  Each output element's K accumulation
// order is the same whatever the rank or tile, so the per-rank projections are
// bit-identical to the matching columns of the full (P = 1) projection.
#include <cuda.h>

#include "h3_device.cuh"
#include "h3_internal.h"

namespace h3 {

constexpr int kProjThreads = 192;

struct ProjTraits {
    static constexpr int BM = 128;   // tokens per tile (TMEM lanes)
    static constexpr int BN = 256;   // output features per tile
    static constexpr int BK = 128;   // bytes (= E4M3 elements) per stage along K
    static constexpr int STAGES = 4;
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = STAGES * A_BYTES;
    static constexpr int OFF_BAR = OFF_B + STAGES * B_BYTES;
    static constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;
    static constexpr int ACC_COLS = BN;  // fp32 accumulator columns per tile
    // kind::f8f6f4: D = f32 (bit 4), A = B = E4M3 (format 0), K-major, N >> 3, M >> 4
    static constexpr uint32_t IDESC =
        (1u << 4) | (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(BM >> 4) << 24);
    static_assert(SMEM_BYTES <= 232448, "shared memory per block");
};

enum : int { PB_FULL = 0, PB_EMPTY = 4, PB_ACC = 8, PB_ACCFREE = 10, PB_DRAIN = 12, PB_COUNT = 13 };

struct ProjParams {
    __nv_bfloat16* out[3];  // q, k, v: [S][Nr] bf16
    int S;
    int Nr;                 // inner / P: output features per part for this rank
    int wrow0;              // rank * Nr
    int inner;
    int n_kblocks;
    int tiles_per_part;
    int n_tiles_n;          // 3 * tiles_per_part
    int n_tiles;            // n_tiles_n * token tiles
    float scale;
    unsigned long long wait_limit_ns;
    DeviceStatus* status;
};

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t smem_dst, const void* tmap, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void proj_drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) break;
    }
}

__global__ void __launch_bounds__(kProjThreads, 1)
    qkv_proj_fp8_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                        const ProjParams p) {
    using T = ProjTraits;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - raw);
    const uint32_t bar0 = sbase + T::OFF_BAR;
    auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + T::OFF_BAR + 8 * PB_COUNT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + T::OFF_BAR + 8 * PB_COUNT + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nk = p.n_kblocks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < T::STAGES; ++s) {
            mbar_init(bar(PB_FULL + s), 1);
            mbar_init(bar(PB_EMPTY + s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar(PB_ACC + a), 1);
            mbar_init(bar(PB_ACCFREE + a), 4);  // one elected lane per epilogue warp
        }
        mbar_init(bar(PB_DRAIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc<512>(smem_u32(tmem_slot));
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl ctl{abort_flag, p.wait_limit_ns, p.status, kTagQkvProj};
    const uint32_t sA = sbase + T::OFF_A, sB = sbase + T::OFF_B;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int it = 0;   // position in the smem ring, continuous across tiles
            int last = -1;
            bool ok = true;
            for (int tile = blockIdx.x; tile < p.n_tiles && ok; tile += gridDim.x) {
                const int nt = tile % p.n_tiles_n, mt = tile / p.n_tiles_n;
                const int part = nt / p.tiles_per_part, ntile = nt - part * p.tiles_per_part;
                const int wrow = part * p.inner + p.wrow0 + ntile * T::BN;
                const int m0 = mt * T::BM;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = it % T::STAGES, u = it / T::STAGES;
                    if (u > 0 && !mbar_wait(bar(PB_EMPTY + s), (u - 1) & 1, ctl, 1)) { ok = false; break; }
                    mbar_arrive_expect_tx(bar(PB_FULL + s), T::A_BYTES + T::B_BYTES);
                    tma_load_2d(sA + s * T::A_BYTES, &tmX, bar(PB_FULL + s), kb * T::BK, m0);
                    tma_load_2d(sB + s * T::B_BYTES, &tmW, bar(PB_FULL + s), kb * T::BK, wrow);
                    last = it;
                }
            }
            if (*abort_flag) {
                for (int i = last; i >= 0 && i > last - T::STAGES; --i)
                    proj_drain_wait(bar(PB_FULL + i % T::STAGES), (i / T::STAGES) & 1, p.wait_limit_ns);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint64_t dA = smem_desc_sw128(sA, 16, 1024);
            const uint64_t dB = smem_desc_sw128(sB, 16, 1024);
            constexpr uint64_t kStageA = T::A_BYTES >> 4, kStageB = T::B_BYTES >> 4;
            bool ok = true;
            int it = 0, n_local = 0;
            for (int tile = blockIdx.x; tile < p.n_tiles && ok; tile += gridDim.x, ++n_local) {
                const int acc = n_local & 1, use = n_local >> 1;
                if (use > 0 && !mbar_wait(bar(PB_ACCFREE + acc), (use - 1) & 1, ctl, 11)) { ok = false; break; }
                tc_fence_after_sync();
                const uint32_t d = tmem + acc * T::ACC_COLS;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = it % T::STAGES, u = it / T::STAGES;
                    if (!mbar_wait(bar(PB_FULL + s), u & 1, ctl, 10)) { ok = false; break; }
                    tc_fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < T::BK / 32; ++kk)  // K = 32 bytes per MMA
                        mma_f8(d, dA + s * kStageA + kk * 2, dB + s * kStageB + kk * 2, T::IDESC,
                               (kb > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(bar(PB_EMPTY + s));  // this stage may be refilled
                }
                if (ok) mma_commit(bar(PB_ACC + acc));
            }
            if (!ok) {
                mma_commit(bar(PB_DRAIN));
                proj_drain_wait(bar(PB_DRAIN), 0, p.wait_limit_ns);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int wq = warp & 3;  // TMEM lane quarter of this warp
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        int n_local = 0;
        for (int tile = blockIdx.x; tile < p.n_tiles; tile += gridDim.x, ++n_local) {
            const int acc = n_local & 1, use = n_local >> 1;
            if (!__all_sync(0xffffffffu, mbar_wait(bar(PB_ACC + acc), use & 1, ctl, 20))) break;
            tc_fence_after_sync();
            const int nt = tile % p.n_tiles_n, mt = tile / p.n_tiles_n;
            const int part = nt / p.tiles_per_part, ntile = nt - part * p.tiles_per_part;
            const int row = mt * T::BM + wq * 32 + lane;
            __nv_bfloat16* base = part == 0 ? p.out[0] : (part == 1 ? p.out[1] : p.out[2]);
            __nv_bfloat16* dst = base + static_cast<size_t>(row) * p.Nr + ntile * T::BN;
            const int cols = min(T::BN, p.Nr - ntile * T::BN);  // multiple of 8
#pragma unroll 1
            for (int c = 0; c < T::BN / 32; ++c) {
                float a[32];
                tmem_ld32(lane_addr + acc * T::ACC_COLS + 32 * c, a);
                if (row < p.S && 32 * c < cols &&
                    in_bounds(p.status, static_cast<size_t>(row) * p.Nr + ntile * T::BN + 32 * c,
                              8ull * min(4, (cols - 32 * c) / 8), static_cast<unsigned long long>(p.S) * p.Nr,
                              kTagQkvProj, 1)) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
                    const int nv = min(4, (cols - 32 * c) / 8);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        if (v < nv) {
                            uint4 wv;
                            wv.x = pack_bf16x2(a[8 * v + 0] * p.scale, a[8 * v + 1] * p.scale);
                            wv.y = pack_bf16x2(a[8 * v + 2] * p.scale, a[8 * v + 3] * p.scale);
                            wv.z = pack_bf16x2(a[8 * v + 4] * p.scale, a[8 * v + 5] * p.scale);
                            wv.w = pack_bf16x2(a[8 * v + 6] * p.scale, a[8 * v + 7] * p.scale);
                            d4[v] = wv;
                        }
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(PB_ACCFREE + acc));
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<512>(tmem);
    }
}

int launch_qkv_proj_fp8(const void* x, const void* w, float scale, void* q_out, void* k_out, void* v_out, int S,
                        int hidden, int inner, int P, int rank, cudaStream_t stream) {
    using T = ProjTraits;
    {
        const int rc = ensure_smem_attr(reinterpret_cast<const void*>(qkv_proj_fp8_kernel), T::SMEM_BYTES);
        if (rc != H3ATTN_OK) return rc;
    }
    CUtensorMap mx, mw;
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(hidden), static_cast<cuuint64_t>(S)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(hidden)};
        const cuuint32_t box[2] = {T::BK, T::BM};
        const cuuint32_t estr[2] = {1, 1};
        int rc = encode_tensor_map(&mx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, x, dims, strides, box, estr,
                                   CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc != H3ATTN_OK) return rc;
    }
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(hidden), static_cast<cuuint64_t>(3) * inner};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(hidden)};
        const cuuint32_t box[2] = {T::BK, T::BN};
        const cuuint32_t estr[2] = {1, 1};
        int rc = encode_tensor_map(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, w, dims, strides, box, estr,
                                   CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc != H3ATTN_OK) return rc;
    }
    ProjParams prm;
    prm.out[0] = static_cast<__nv_bfloat16*>(q_out);
    prm.out[1] = static_cast<__nv_bfloat16*>(k_out);
    prm.out[2] = static_cast<__nv_bfloat16*>(v_out);
    prm.S = S;
    prm.Nr = inner / P;
    prm.wrow0 = rank * (inner / P);
    prm.inner = inner;
    prm.n_kblocks = (hidden + T::BK - 1) / T::BK;
    prm.tiles_per_part = (prm.Nr + T::BN - 1) / T::BN;
    prm.n_tiles_n = 3 * prm.tiles_per_part;
    prm.n_tiles = prm.n_tiles_n * ((S + T::BM - 1) / T::BM);
    prm.scale = scale;
    prm.wait_limit_ns = wait_limit_ns();
    int rc = device_status_ptr(&prm.status);
    if (rc != H3ATTN_OK) return rc;
    int n_sm = 0;
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    const unsigned grid = static_cast<unsigned>(min(prm.n_tiles, n_sm));
    qkv_proj_fp8_kernel<<<grid, kProjThreads, T::SMEM_BYTES, stream>>>(mx, mw, prm);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? H3ATTN_OK : cuda_fail(e);
}

}  // namespace h3
