// h3attn_abi.cu -- the extern "C" entry points declared in include/h3attn.h:
// argument checking on the host, then a launch on the caller's stream.
// Nothing here computes; every step of the path runs in the kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <nvtx3/nvToolsExt.h>

#include <cstdint>
#include <cstdlib>
#include <cmath>
#include <atomic>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "h3_device.cuh"
#include "h3_internal.h"

namespace h3 {

constexpr int kMaxDevices = 64;

// One status word per device, and the slot the take kernel copies it into.
__device__ DeviceStatus g_status;
__device__ unsigned long long g_status_taken;

static int status_ptrs(DeviceStatus** status, unsigned long long** taken) {
    static DeviceStatus* cache[kMaxDevices] = {};
    static unsigned long long* cache_taken[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return H3ATTN_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == nullptr) {
        void* p = nullptr;
        void* t = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_status)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaGetSymbolAddress(&t, g_status_taken)) != cudaSuccess) return cuda_fail(e);
        cache[dev] = static_cast<DeviceStatus*>(p);
        cache_taken[dev] = static_cast<unsigned long long*>(t);
    }
    *status = cache[dev];
    if (taken != nullptr) *taken = cache_taken[dev];
    return H3ATTN_OK;
}

int device_status_ptr(DeviceStatus** out) { return status_ptrs(out, nullptr); }

// Read and clear the status word in one atomic exchange, so an error that a
// kernel on another stream records at the same moment is either taken whole
// now or left for the next read -- never erased unseen.
__global__ void status_take_kernel(DeviceStatus* st, unsigned long long* taken) {
    *taken = atomicExch(&st->word, 0ull);
}

int ensure_smem_attr(const void* kernel, int bytes) {
    constexpr int kMaxDevices = 64;
    constexpr int kMaxKernels = 8;
    static const void* done[kMaxDevices][kMaxKernels] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return H3ATTN_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < kMaxKernels; ++i) {
        if (done[dev][i] == kernel) return H3ATTN_OK;
        if (done[dev][i] == nullptr) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
            if (e != cudaSuccess) return cuda_fail(e);
            done[dev][i] = kernel;
            return H3ATTN_OK;
        }
    }
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return e == cudaSuccess ? H3ATTN_OK : cuda_fail(e);
}

static thread_local int t_last_cuda_error = 0;
// Diagnostic info of the last device error taken on each device.
static std::atomic<unsigned long long> g_last_info[kMaxDevices];

int cuda_fail(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return H3ATTN_ERR_CUDA;
}

unsigned long long wait_limit_ns() {
    static unsigned long long v = [] {
        const char* s = std::getenv("H3ATTN_WAIT_LIMIT_NS");
        if (s != nullptr) {
            const unsigned long long x = std::strtoull(s, nullptr, 10);
            if (x >= 1000ull && x <= 60000000000ull) return x;
        }
        return 2000000000ull;
    }();
    return v;
}

int encode_tensor_map(CUtensorMap* m, CUtensorMapDataType dtype, unsigned rank, const void* base,
                      const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box,
                      const cuuint32_t* elem_strides, CUtensorMapSwizzle swizzle) {
    using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static EncodeFn fn = nullptr;
    static std::once_flag once;
    static cudaError_t lookup_err = cudaSuccess;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        lookup_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (lookup_err == cudaSuccess && q == cudaDriverEntryPointSuccess) fn = reinterpret_cast<EncodeFn>(p);
        else if (lookup_err == cudaSuccess) lookup_err = cudaErrorNotSupported;
    });
    if (fn == nullptr) return cuda_fail(lookup_err);
    const CUresult r = fn(m, dtype, rank, const_cast<void*>(base), dims, strides_bytes, box, elem_strides,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
    return H3ATTN_OK;
}

// Failure-detection self-test: a wait on an mbarrier that nothing arrives on.
__global__ void selftest_wait_kernel(unsigned long long limit_ns, DeviceStatus* status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const WaitCtl ctl{&abort_flag, limit_ns, status, kTagSelftest};
    if (threadIdx.x == 0) (void)mbar_wait(smem_u32(&bar), 0, ctl, 1);
}

int launch_selftest_wait(unsigned long long limit_ns, cudaStream_t stream) {
    DeviceStatus* status = nullptr;
    const int rc = device_status_ptr(&status);
    if (rc != H3ATTN_OK) return rc;
    selftest_wait_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? H3ATTN_OK : cuda_fail(e);
}

// ----------------------------------------------------------------------------
// Host-side checks
// ----------------------------------------------------------------------------
// The norm kernel finds a head's group by multiplying with ceil(2^32 / (H/P))
// and shifting; that is exact while (H - 1) * (H/P) < 2^32, which every H up
// to 65535 satisfies.
constexpr int kMaxNormHeads = 65535;

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// The kernels are built for sm_103a only; refuse anything else up front so a
// wrong device fails with a clear code instead of a launch error.  Then every
// buffer pointer must be memory the current device's kernels can address:
// device memory of this device, or managed memory.  A host pointer, or
// device memory of another GPU, is refused with H3ATTN_ERR_ARG before
// anything is launched (null entries are optional buffers and are skipped).
static int check_device(std::initializer_list<const void*> ptrs = {}) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return cuda_fail(e);
    if (major != 10 || minor != 3) return H3ATTN_ERR_UNSUPPORTED_DEVICE;
    for (const void* p : ptrs) {
        if (p == nullptr) continue;
        cudaPointerAttributes a;
        e = cudaPointerGetAttributes(&a, p);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();  // an unknown pointer is an argument error, not a sticky CUDA error
            return H3ATTN_ERR_ARG;
        }
        if (a.type == cudaMemoryTypeManaged) continue;
        if (a.type != cudaMemoryTypeDevice || a.device != dev) return H3ATTN_ERR_ARG;
    }
    return H3ATTN_OK;
}

static int check_layout_args(const void* in, const void* out, int S, int H, int D, int P) {
    if (in == nullptr || out == nullptr) return H3ATTN_ERR_ARG;
    if (!aligned16(in) || !aligned16(out)) return H3ATTN_ERR_ARG;
    if (S < 1 || H < 1 || P < 1 || (D != 64 && D != 128)) return H3ATTN_ERR_SHAPE;
    if (S % P != 0 || H % P != 0) return H3ATTN_ERR_SHAPE;
    const uint64_t elems = static_cast<uint64_t>(S) * H * D;
    if (elems / 8 >= (1ull << 32)) return H3ATTN_ERR_SHAPE;
    if (overlap(in, elems * 2, out, elems * 2)) return H3ATTN_ERR_ALIAS;
    return H3ATTN_OK;
}

// NVTX range around each entry point (header-only NVTX v3: a no-op unless a
// profiler is attached), so timelines show which library call issued a kernel.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

}  // namespace h3

using namespace h3;

extern "C" {

int h3attn_version(void) { return H3ATTN_VERSION; }

int h3attn_build_flags(void) { return H3ATTN_DEBUG_CHECKS ? H3ATTN_BUILD_DEBUG_CHECKS : 0; }

int h3attn_last_cuda_error(void) { return t_last_cuda_error; }

unsigned long long h3attn_last_device_error_info(void) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return 0;
    }
    return g_last_info[dev].load();
}

const char* h3attn_strerror(int code) {
    switch (code) {
        case H3ATTN_OK: return "ok";
        case H3ATTN_ERR_ARG: return "invalid argument (null or misaligned pointer, or bad scalar)";
        case H3ATTN_ERR_SHAPE: return "unsupported or inconsistent sizes";
        case H3ATTN_ERR_ALIAS: return "output overlaps an input";
        case H3ATTN_ERR_CUDA: return "CUDA call failed";
        case H3ATTN_ERR_DEVICE_TIMEOUT: return "a kernel gave up on a pipeline wait (device timeout)";
        case H3ATTN_ERR_UNSUPPORTED_DEVICE: return "current device is not sm_103";
        case H3ATTN_ERR_DEVICE_BOUNDS: return "a kernel's index check failed and the access was skipped (debug-check build)";
        default: return "unknown status";
    }
}

int h3attn_qk_norm_rope(const void* q, const void* k, void* q_out, void* k_out, float* dbg_fp32,
                        const float* w_q, const float* w_k, const int32_t* pos, int B, int S, int H, int D,
                        int d_t, int d_h, int d_w, float eps, float theta, void* stream) {
    const NvtxRange nvtx_range("h3attn_qk_norm_rope");
    if (!q || !k || !q_out || !k_out || !w_q || !w_k || !pos) return H3ATTN_ERR_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(q_out) || !aligned16(k_out) || !aligned16(w_q) ||
        !aligned16(w_k) || (dbg_fp32 && !aligned16(dbg_fp32)))
        return H3ATTN_ERR_ARG;
    if (!(eps >= 0.0f) || !(theta > 0.0f)) return H3ATTN_ERR_ARG;
    if (B < 1 || S < 1 || H < 1 || H > kMaxNormHeads || (D != 64 && D != 128)) return H3ATTN_ERR_SHAPE;
    if (d_t < 0 || d_h < 0 || d_w < 0 || (d_t | d_h | d_w) & 1 || d_t + d_h + d_w != D) return H3ATTN_ERR_SHAPE;
    if (static_cast<uint64_t>(B) * S >= (1ull << 31)) return H3ATTN_ERR_SHAPE;
    const size_t bytes = static_cast<size_t>(B) * S * H * D * 2;
    if (q_out != q && overlap(q, bytes, q_out, bytes)) return H3ATTN_ERR_ALIAS;
    if (k_out != k && overlap(k, bytes, k_out, bytes)) return H3ATTN_ERR_ALIAS;
    if (overlap(q_out, bytes, k_out, bytes)) return H3ATTN_ERR_ALIAS;
    if (overlap(q_out, bytes, k, bytes) || overlap(k_out, bytes, q, bytes)) return H3ATTN_ERR_ALIAS;
    if (dbg_fp32 && (overlap(dbg_fp32, bytes * 4, q_out, bytes) || overlap(dbg_fp32, bytes * 4, k_out, bytes)))
        return H3ATTN_ERR_ALIAS;
    int rc = check_device({q, k, q_out, k_out, dbg_fp32, w_q, w_k, pos});
    if (rc != H3ATTN_OK) return rc;
    return launch_norm_rope(q, k, q_out, k_out, dbg_fp32, w_q, w_k, pos, B, S, H, D, d_t, d_h, d_w, eps,
                            static_cast<double>(theta), 1, static_cast<cudaStream_t>(stream));
}

int h3attn_qk_norm_rope_seq2head(const void* q, const void* k, void* qh_out, void* kh_out, float* dbg_fp32,
                                 const float* w_q, const float* w_k, const int32_t* pos, int S, int H, int D,
                                 int P, int d_t, int d_h, int d_w, float eps, float theta, void* stream) {
    const NvtxRange nvtx_range("h3attn_qk_norm_rope_seq2head");
    if (!q || !k || !qh_out || !kh_out || !w_q || !w_k || !pos) return H3ATTN_ERR_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(qh_out) || !aligned16(kh_out) || !aligned16(w_q) ||
        !aligned16(w_k) || (dbg_fp32 && !aligned16(dbg_fp32)))
        return H3ATTN_ERR_ARG;
    if (!(eps >= 0.0f) || !(theta > 0.0f)) return H3ATTN_ERR_ARG;
    if (S < 1 || H < 1 || H > kMaxNormHeads || P < 1 || (D != 64 && D != 128)) return H3ATTN_ERR_SHAPE;
    if (S % P != 0 || H % P != 0) return H3ATTN_ERR_SHAPE;
    if (d_t < 0 || d_h < 0 || d_w < 0 || (d_t | d_h | d_w) & 1 || d_t + d_h + d_w != D) return H3ATTN_ERR_SHAPE;
    if (static_cast<uint64_t>(S) * H * D / 8 >= (1ull << 32)) return H3ATTN_ERR_SHAPE;
    const size_t bytes = static_cast<size_t>(S) * H * D * 2;
    // the output is a permutation of the input, so it may not share memory with it
    if (overlap(q, bytes, qh_out, bytes) || overlap(k, bytes, kh_out, bytes) || overlap(q, bytes, kh_out, bytes) ||
        overlap(k, bytes, qh_out, bytes) || overlap(qh_out, bytes, kh_out, bytes))
        return H3ATTN_ERR_ALIAS;
    if (dbg_fp32 && (overlap(dbg_fp32, bytes * 4, qh_out, bytes) || overlap(dbg_fp32, bytes * 4, kh_out, bytes)))
        return H3ATTN_ERR_ALIAS;
    int rc = check_device({q, k, qh_out, kh_out, dbg_fp32, w_q, w_k, pos});
    if (rc != H3ATTN_OK) return rc;
    return launch_norm_rope(q, k, qh_out, kh_out, dbg_fp32, w_q, w_k, pos, 1, S, H, D, d_t, d_h, d_w, eps,
                            static_cast<double>(theta), P, static_cast<cudaStream_t>(stream));
}

int h3attn_forward(const void* q, const void* k, const void* v, void* o, int B, int S, int H_buf, int D,
                   int head_begin, int head_count, const int32_t* kv_len, float scale, void* stream) {
    const NvtxRange nvtx_range("h3attn_forward");
    if (!q || !k || !v || !o) return H3ATTN_ERR_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return H3ATTN_ERR_ARG;
    if (!(scale == scale)) return H3ATTN_ERR_ARG;  // NaN
    if (B < 1 || S < 1 || H_buf < 1 || (D != 64 && D != 128)) return H3ATTN_ERR_SHAPE;
    if (head_begin < 0 || head_count < 1 || head_begin + head_count > H_buf || head_count > 65535)
        return H3ATTN_ERR_SHAPE;
    if (kv_len != nullptr) {
        // kv_len is read here, on the host: refuse device memory before touching it.
        // Host memory (pageable or pinned) reports success with a host type; if
        // the query itself fails there is no usable CUDA device, so the pointer
        // cannot be device memory (the device check below then fails the call).
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, kv_len) == cudaSuccess) {
            if (a.type == cudaMemoryTypeDevice) return H3ATTN_ERR_ARG;
        } else {
            (void)cudaGetLastError();
        }
        for (int b = 0; b < B; ++b)
            if (kv_len[b] < 1 || kv_len[b] > S) return H3ATTN_ERR_SHAPE;
    }
    const size_t item = static_cast<size_t>(S) * H_buf * D * 2;
    const size_t bytes = item * B;
    if (overlap(o, bytes, q, bytes) || overlap(o, bytes, k, bytes) || overlap(o, bytes, v, bytes))
        return H3ATTN_ERR_ALIAS;
    int rc = check_device({q, k, v, o});
    if (rc != H3ATTN_OK) return rc;
    const float sc = scale > 0.0f ? scale : 1.0f / std::sqrt(static_cast<float>(D));
    for (int b = 0; b < B; ++b) {
        const size_t off = item * b;
        rc = launch_attention(static_cast<const char*>(q) + off, static_cast<const char*>(k) + off,
                              static_cast<const char*>(v) + off, static_cast<char*>(o) + off, S, H_buf, D,
                              head_begin, head_count, kv_len ? kv_len[b] : S, sc,
                              static_cast<cudaStream_t>(stream));
        if (rc != H3ATTN_OK) return rc;
    }
    return H3ATTN_OK;
}

int h3attn_seq2head(const void* in, void* out, int S, int H, int D, int P, void* stream) {
    const NvtxRange nvtx_range("h3attn_seq2head");
    int rc = check_layout_args(in, out, S, H, D, P);
    if (rc != H3ATTN_OK) return rc;
    if ((rc = check_device({in, out})) != H3ATTN_OK) return rc;
    return launch_seq2head(in, out, S, H, D, P, static_cast<cudaStream_t>(stream));
}

int h3attn_head2seq(const void* in, void* out, int S, int H, int D, int P, void* stream) {
    const NvtxRange nvtx_range("h3attn_head2seq");
    int rc = check_layout_args(in, out, S, H, D, P);
    if (rc != H3ATTN_OK) return rc;
    if ((rc = check_device({in, out})) != H3ATTN_OK) return rc;
    return launch_head2seq(in, out, S, H, D, P, static_cast<cudaStream_t>(stream));
}

int h3attn_head2seq_heads(const void* in_group, void* out, int S, int H, int D, int P, int group,
                          int head_begin, int head_count, void* stream) {
    const NvtxRange nvtx_range("h3attn_head2seq_heads");
    if (in_group == nullptr || out == nullptr) return H3ATTN_ERR_ARG;
    if (!aligned16(in_group) || !aligned16(out)) return H3ATTN_ERR_ARG;
    if (S < 1 || H < 1 || P < 1 || (D != 64 && D != 128) || H % P != 0) return H3ATTN_ERR_SHAPE;
    const int Hp = H / P;
    if (group < 0 || group >= P || head_begin < 0 || head_count < 1 || head_begin + head_count > Hp)
        return H3ATTN_ERR_SHAPE;
    const uint64_t elems = static_cast<uint64_t>(S) * H * D;
    if (elems / 8 >= (1ull << 32)) return H3ATTN_ERR_SHAPE;
    const size_t in_bytes = static_cast<size_t>(S) * Hp * D * 2;
    if (overlap(in_group, in_bytes, out, elems * 2)) return H3ATTN_ERR_ALIAS;
    int rc = check_device({in_group, out});
    if (rc != H3ATTN_OK) return rc;
    return launch_head2seq_heads(in_group, out, S, H, D, P, group, head_begin, head_count,
                                 static_cast<cudaStream_t>(stream));
}

int h3attn_qkv_proj_fp8(const void* x, const void* w, float scale, void* q_out, void* k_out, void* v_out, int S,
                        int hidden, int inner, int P, int rank, void* stream) {
    const NvtxRange nvtx_range("h3attn_qkv_proj_fp8");
    if (!x || !w || !q_out || !k_out || !v_out) return H3ATTN_ERR_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(q_out) || !aligned16(k_out) || !aligned16(v_out))
        return H3ATTN_ERR_ARG;
    if (!(scale == scale)) return H3ATTN_ERR_ARG;
    if (S < 1 || hidden < 16 || hidden % 16 != 0 || inner < 1 || P < 1 || inner % P != 0) return H3ATTN_ERR_SHAPE;
    if (rank < 0 || rank >= P || (inner / P) % 8 != 0) return H3ATTN_ERR_SHAPE;
    const size_t xb = static_cast<size_t>(S) * hidden, wb = static_cast<size_t>(3) * inner * hidden;
    const size_t ob = static_cast<size_t>(S) * (inner / P) * 2;
    const void* outs[3] = {q_out, k_out, v_out};
    for (int i = 0; i < 3; ++i) {
        if (overlap(outs[i], ob, x, xb) || overlap(outs[i], ob, w, wb)) return H3ATTN_ERR_ALIAS;
        for (int j = i + 1; j < 3; ++j)
            if (overlap(outs[i], ob, outs[j], ob)) return H3ATTN_ERR_ALIAS;
    }
    int rc = check_device({x, w, q_out, k_out, v_out});
    if (rc != H3ATTN_OK) return rc;
    return launch_qkv_proj_fp8(x, w, scale, q_out, k_out, v_out, S, hidden, inner, P, rank,
                               static_cast<cudaStream_t>(stream));
}

int h3attn_get_device_status(void* stream) {
    static std::mutex mu[kMaxDevices];  // one take in flight per device: the copy-out slot is shared
    DeviceStatus* st = nullptr;
    unsigned long long* taken = nullptr;
    int rc = status_ptrs(&st, &taken);
    if (rc != H3ATTN_OK) return rc;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned long long word = 0;
    {
        std::lock_guard<std::mutex> lock(mu[dev]);
        status_take_kernel<<<1, 1, 0, s>>>(st, taken);
        if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaMemcpyAsync(&word, taken, sizeof(word), cudaMemcpyDeviceToHost, s)) != cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e);
    }
    if (word != 0) g_last_info[dev].store(status_info(word));
    return status_code(word);
}

int h3attn_selftest_wait_timeout(unsigned long long limit_ns, void* stream) {
    if (limit_ns < 1 || limit_ns > 10000000000ull) return H3ATTN_ERR_ARG;
    int rc = check_device();
    if (rc != H3ATTN_OK) return rc;
    return launch_selftest_wait(limit_ns, static_cast<cudaStream_t>(stream));
}

int h3attn_selftest_bounds(void* buf, unsigned long long bytes, void* stream) {
    const NvtxRange nvtx_range("h3attn_selftest_bounds");
    if (!H3ATTN_DEBUG_CHECKS) return H3ATTN_ERR_ARG;
    if (buf == nullptr || !aligned16(buf) || bytes < 1024) return H3ATTN_ERR_ARG;
    int rc = check_device({buf});
    if (rc != H3ATTN_OK) return rc;
    return launch_selftest_bounds(buf, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
