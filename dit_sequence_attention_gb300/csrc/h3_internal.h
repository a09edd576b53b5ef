// h3_internal.h -- host-side declarations shared by the kernel files and the
// C-ABI front end (h3attn_abi.cu).  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "h3attn.h"

namespace h3 {

struct DeviceStatus;

// Address of the current device's status word (looked up once per device).
int device_status_ptr(DeviceStatus** out);

// Records `e` as this thread's last CUDA error and returns H3ATTN_ERR_CUDA.
int cuda_fail(cudaError_t e);

// Sets the kernel's dynamic shared-memory limit once per device (the
// attribute is per device; a process may drive several GPUs).
int ensure_smem_attr(const void* kernel, int bytes);

// Per-wait time limit handed to the kernels (nanoseconds).  2 s unless the
// environment variable H3ATTN_WAIT_LIMIT_NS overrides it.
unsigned long long wait_limit_ns();

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda
// link dependency, so the library also loads on machines without a driver).
int encode_tensor_map(CUtensorMap* m, CUtensorMapDataType dtype, unsigned rank, const void* base,
                      const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box,
                      const cuuint32_t* elem_strides, CUtensorMapSwizzle swizzle);

int launch_attention(const void* q, const void* k, const void* v, void* o, int S, int H_buf, int D, int head_begin,
                     int head_count, int kv_len, float scale, cudaStream_t stream);

int launch_norm_rope(const void* q, const void* k, void* q_out, void* k_out, float* dbg, const float* w_q,
                     const float* w_k, const int32_t* pos, int B, int S, int H, int D, int d_t, int d_h, int d_w,
                     float eps, double theta, int P, cudaStream_t stream);

int launch_seq2head(const void* in, void* out, int S, int H, int D, int P, cudaStream_t stream);
int launch_head2seq(const void* in, void* out, int S, int H, int D, int P, cudaStream_t stream);
int launch_head2seq_heads(const void* in_group, void* out, int S, int H, int D, int P, int g, int j0, int jc,
                          cudaStream_t stream);

int launch_qkv_proj_fp8(const void* x, const void* w, float scale, void* q_out, void* k_out, void* v_out, int S,
                        int hidden, int inner, int P, int rank, cudaStream_t stream);

int launch_selftest_wait(unsigned long long limit_ns, cudaStream_t stream);
int launch_selftest_bounds(void* buf, cudaStream_t stream);

}  // namespace h3
