/*
 * h3attn.h -- C ABI of the GB300 (sm_103a) attention hot path of a
 * MiniMax-H3-style video+audio DiT block:
 *
 *   QK-RMSNorm + 3-axis RoPE  ->  Ulysses seq->head layout  ->  exact masked
 *   multi-head attention over the packed sequence  ->  head->seq layout.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Tensors are row-major, token-major: [B][S][H][D] (batch, packed sequence,
 *    head, head_dim), bf16 elements stored as raw 16-bit words.  head_dim D is
 *    64 or 128; the head count is a runtime value, which is how a caller hands
 *    the kernel a buffer that holds only 56/P heads (the diffusers TP PR
 *    reshapes attention by the fixed head_dim and lets the head count follow).
 *  - Every tensor pointer is a DEVICE pointer of the current device (or
 *    managed memory), 16-byte aligned; anything else (a host pointer, memory
 *    of another GPU) is refused with H3ATTN_ERR_ARG before any launch.  The
 *    caller owns all buffers; the library allocates no device memory per call.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls only enqueue work and return; nothing synchronises except
 *    h3attn_get_device_status().
 *  - Return value: H3ATTN_OK (0) or a negative H3ATTN_ERR_* code.  Arguments
 *    are checked on the host before anything is launched; a rejected call
 *    enqueues nothing.  No call traps or aborts the process.
 *  - Device errors (a pipeline wait that ran out of time; in the debug-check
 *    build libh3attn_debug.so, an index check that failed) are recorded in a
 *    device status word and reported by h3attn_get_device_status().
 */
#ifndef H3ATTN_H
#define H3ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define H3ATTN_VERSION 1

#if defined(__GNUC__)
#define H3ATTN_API __attribute__((visibility("default")))
#else
#define H3ATTN_API
#endif

enum h3attn_status {
    H3ATTN_OK = 0,
    H3ATTN_ERR_ARG = -1,            /* null/misaligned pointer, bad scalar (eps < 0, theta <= 0, ...) */
    H3ATTN_ERR_SHAPE = -2,          /* unsupported or inconsistent sizes */
    H3ATTN_ERR_ALIAS = -3,          /* output overlaps an input where that is not allowed */
    H3ATTN_ERR_CUDA = -4,           /* a CUDA runtime/driver call failed (see h3attn_last_cuda_error) */
    H3ATTN_ERR_DEVICE_TIMEOUT = -5, /* a kernel gave up on a pipeline wait (device status word) */
    H3ATTN_ERR_UNSUPPORTED_DEVICE = -6, /* current device is not an sm_103 (GB300-class) GPU */
    H3ATTN_ERR_DEVICE_BOUNDS = -7   /* debug-check builds: a kernel computed an index outside its buffer
                                       and skipped that access (device status word) */
};

/* Bits of h3attn_build_flags(). */
#define H3ATTN_BUILD_DEBUG_CHECKS 1 /* kernels check every computed global index before the access */

/*
 * h3attn_qk_norm_rope -- fused QK-RMSNorm and three-axis rotary embedding.
 *
 * Defined by "[feat] Tensor parallelism for MiniMax-H3" (diffusers PR #14609),
 * PR description: the QK-norms are head_dim-shaped and applied after the head
 * split; the rotary embedding uses real sin/cos, broadcasts over the head axis,
 * and takes its angle as inv_freq times the position (loader-bug comment on
 * the same page).  For every batch b, token s, head h and separately for q and k:
 *     y[d]  = x[d] / sqrt(mean_e x[e]^2 + eps) * w[d]            (fp32)
 *     axis a in (t, h, w) owns dims [off_a, off_a + d_a), off = (0, d_t, d_t + d_h);
 *     pair i of axis a = dims (off_a + 2i, off_a + 2i + 1), angle = pos[s][a] * theta^(-2i/d_a);
 *     (y0, y1) -> (y0 cos - y1 sin, y0 sin + y1 cos)
 * then one round-to-nearest-even to bf16.  v is not touched.
 *
 *   q, k        [B][S][H][D] bf16 inputs.
 *   q_out,k_out [B][S][H][D] bf16 outputs; may equal q / k (in place), must
 *               not partially overlap them.
 *   dbg_fp32    NULL, or [2][B][S][H][D] fp32 receiving the unrounded q then k
 *               results (test aid).
 *   w_q, w_k    [D] fp32 norm weights (shared by all heads).
 *   pos         [S][3] int32 (t, h, w) positions, shared by all batch items.
 *   d_t+d_h+d_w == D, each even.  eps >= 0, theta > 0.  1 <= H <= 65535,
 *   B * S < 2^31 (H3ATTN_ERR_SHAPE otherwise).
 */
H3ATTN_API int h3attn_qk_norm_rope(const void* q, const void* k, void* q_out, void* k_out, float* dbg_fp32,
                        const float* w_q, const float* w_k, const int32_t* pos, int B, int S, int H, int D,
                        int d_t, int d_h, int d_w, float eps, float theta, void* stream);

/*
 * h3attn_qk_norm_rope_seq2head -- h3attn_qk_norm_rope followed by
 * h3attn_seq2head of its q and k outputs, in one pass: the results are
 * written straight into the Ulysses head-sharded layout.  The README of
 * "buqi-minimax-h3-multigpu" ("How it works") counts the transpose+copy steps
 * around the exchange as a cost worth removing; here the normalised q and k
 * skip their token-major round trip through HBM.
 *   q, k          [S][H][D] bf16 (one batch item; the P sequence shards).
 *   qh_out,kh_out [P][S][H/P][D] bf16, bit-identical to
 *                 seq2head(qk_norm_rope(q, k)); must not overlap q or k.
 *   dbg_fp32      NULL, or [2][S][H][D] fp32 (token-major, unrounded q then k).
 *   S % P == 0, H % P == 0, 1 <= H <= 65535, S * H * D / 8 < 2^32; other
 *   arguments as h3attn_qk_norm_rope.
 */
H3ATTN_API int h3attn_qk_norm_rope_seq2head(const void* q, const void* k, void* qh_out, void* kh_out,
                                            float* dbg_fp32, const float* w_q, const float* w_k,
                                            const int32_t* pos, int S, int H, int D, int P, int d_t, int d_h,
                                            int d_w, float eps, float theta, void* stream);

/*
 * h3attn_forward -- exact softmax attention for a range of heads.
 *
 * Defined by "buqi-minimax-h3-multigpu" README, sections "On accuracy" and
 * "How it works": every rank evaluates exact full attention over the whole
 * packed sequence for its subset of the 56 heads.  Keys at positions >=
 * kv_len[b] are padding (the sequence is padded to a multiple of 512; see the
 * NKI note in the diffusers TP PR) and get weight exactly zero:
 *     o[b][i][h] = sum_{j < kv_len[b]} softmax_j(scale * <q[b][i][h], k[b][j][h]>) v[b][j][h]
 * for h in [head_begin, head_begin + head_count) and every query row i < S
 * (padded query rows are computed like any other).  bf16 operands, fp32
 * accumulation, the probabilities rounded to bf16 for the PV product, bf16
 * output.  Heads outside the range are not written.
 *
 *   q, k, v, o  [B][S][H_buf][D] bf16; o must not overlap q, k or v.
 *   kv_len      HOST array [B] with 1 <= kv_len[b] <= S, or NULL for all S.
 *               It is read on the host during the call; a device pointer is
 *               refused with H3ATTN_ERR_ARG before it is touched.
 *               Rows >= kv_len[b] of k and v are never read (NaN there is fine).
 *   scale       softmax scale; <= 0 selects 1/sqrt(D); NaN is refused (H3ATTN_ERR_ARG).
 *   B >= 1, S >= 1, 0 <= head_begin, 1 <= head_count <= 65535 and
 *   head_begin + head_count <= H_buf (H3ATTN_ERR_SHAPE otherwise).
 * The per-head result does not depend on head_begin/head_count or on how many
 * heads one call covers: splitting the heads over several calls gives
 * bit-identical output.
 */
H3ATTN_API int h3attn_forward(const void* q, const void* k, const void* v, void* o, int B, int S, int H_buf, int D,
                   int head_begin, int head_count, const int32_t* kv_len, float scale, void* stream);

/*
 * h3attn_seq2head -- Ulysses sequence->head exchange as a single-GPU layout
 * transform ("buqi-minimax-h3-multigpu" README, "How it works": the sequence
 * is row-sharded over P ranks for per-token work; attention needs every row
 * for 56/P heads, so an all-to-all regroups q, k and v by head).
 *     in  [P][S/P][H][D]  (the P sequence shards, i.e. one [S][H][D] tensor)
 *     out [P][S][H/P][D]  out[g][s][j] = in[s / (S/P)][s % (S/P)][g*(H/P) + j]
 * Pure 16-bit word movement (bit-exact).  S % P == 0, H % P == 0, P >= 1.
 * in and out must not overlap.
 */
H3ATTN_API int h3attn_seq2head(const void* in, void* out, int S, int H, int D, int P, void* stream);

/*
 * h3attn_head2seq -- the inverse exchange (the attention output all-to-all,
 * "How it works" of the same README):
 *     in  [P][S][H/P][D]  ->  out [P][S/P][H][D],
 *     out[r][i][g*(H/P) + j] = in[g][r*(S/P) + i][j].
 * head2seq(seq2head(x)) == x bit for bit.  in and out must not overlap.
 */
H3ATTN_API int h3attn_head2seq(const void* in, void* out, int S, int H, int D, int P, void* stream);

/*
 * h3attn_head2seq_heads -- the output exchange for one chunk of one group's
 * heads, so that it can run on a second stream while attention computes the
 * next chunk ("buqi-minimax-h3-multigpu" README, "How it works": attention
 * runs in head chunks and each chunk's output exchange overlaps the next
 * chunk's compute; the result does not depend on the chunk count).
 *   in_group  [S][H/P][D] bf16: head group `group` (0 <= group < P).
 *   out       [S][H][D] bf16; heads group*(H/P) + j for j in
 *             [head_begin, head_begin + head_count) are written, no others.
 *   in_group and out must not overlap.
 */
H3ATTN_API int h3attn_head2seq_heads(const void* in_group, void* out, int S, int H, int D, int P, int group,
                                     int head_begin, int head_count, void* stream);

/*
 * h3attn_qkv_proj_fp8 -- the all-gather exchange variant's projection: the
 * gathered hidden state times only this rank's head rows of qkv_proj
 * ("buqi-minimax-h3-multigpu" README, "How it works": for world sizes up to
 * 4 each rank receives the modulated hidden state and projects it through its
 * own head rows of qkv_proj; slicing the fp8 weight by rows is exact because
 * its scale is one number per tensor).  For part in (q, k, v):
 *     out_part[s][c] = scale * sum_e x[s][e] * w[part*inner + rank*inner/P + c][e]
 *   x       [S][hidden] FP8 E4M3 codes (hidden % 16 == 0).
 *   w       [3*inner][hidden] FP8 E4M3 codes: q rows, then k rows, then v
 *           rows; head h of a part owns rows [h*D, (h+1)*D) of it.
 *   scale   product of the two per-tensor scales (applied in fp32).
 *   q_out, k_out, v_out  [S][inner/P] bf16 each, i.e. [S][H/P][D]: this
 *           rank's heads in the layout h3attn_forward reads.  (inner/P) % 8 == 0.
 *   0 <= rank < P.  FP8 products, fp32 accumulation; the result for a given
 *   (s, part, global column) is bit-identical for every P and rank.
 */
H3ATTN_API int h3attn_qkv_proj_fp8(const void* x, const void* w, float scale, void* q_out, void* k_out,
                                   void* v_out, int S, int hidden, int inner, int P, int rank, void* stream);

/*
 * h3attn_get_device_status -- take the device status word of the current
 * device: a one-thread kernel enqueued on `stream` reads and clears it in one
 * atomic exchange, then the call synchronises `stream` and returns what it
 * read.  Returns H3ATTN_OK, H3ATTN_ERR_DEVICE_TIMEOUT (a kernel gave up on a
 * wait, wrote nothing trustworthy and returned), H3ATTN_ERR_DEVICE_BOUNDS
 * (debug-check builds only: a kernel's index check failed and the access was
 * skipped), or H3ATTN_ERR_CUDA if the launch or synchronisation failed.  The
 * first error recorded since the last take wins.  Errors recorded by kernels
 * on other streams are reported if they landed before the take, and kept for
 * the next call otherwise; none is cleared without being returned.  Calls
 * from several host threads are serialised per device.
 */
H3ATTN_API int h3attn_get_device_status(void* stream);

/* Diagnostic word recorded with the last device error taken on the current
 * device, 0 if none; read after h3attn_get_device_status.  Kernel tag << 32 |
 * site << 16 | low 16 bits of the block index (timeouts) or of the offending
 * index (bounds checks).  Kernel tags: 1 attention, 2 wait self-test, 3 fp8
 * projection, 4 norm/RoPE, 5 seq2head, 6 head2seq, 7 head2seq_heads. */
H3ATTN_API unsigned long long h3attn_last_device_error_info(void);

/* cudaError_t value behind the most recent H3ATTN_ERR_CUDA on this thread. */
H3ATTN_API int h3attn_last_cuda_error(void);

/* Static description of a status code. */
H3ATTN_API const char* h3attn_strerror(int code);

/* H3ATTN_VERSION of the built library. */
H3ATTN_API int h3attn_version(void);

/* H3ATTN_BUILD_* bits the library was compiled with (0 for the release build;
 * H3ATTN_BUILD_DEBUG_CHECKS for libh3attn_debug.so). */
H3ATTN_API int h3attn_build_flags(void);

/*
 * h3attn_selftest_wait_timeout -- failure-detection self-test.  Launches one
 * block whose wait on an mbarrier that nothing ever arrives on uses the same
 * bounded wait as the attention pipeline, with a limit of `limit_ns`
 * nanoseconds (1 <= limit_ns <= 10^10).  The wait runs out, the kernel records
 * H3ATTN_ERR_DEVICE_TIMEOUT and returns; the next h3attn_get_device_status()
 * reports it and the context stays usable.
 */
H3ATTN_API int h3attn_selftest_wait_timeout(unsigned long long limit_ns, void* stream);

/*
 * h3attn_selftest_bounds -- self-test of the device index checks of a
 * debug-check build.  Runs the seq2head kernel on a tiny case (S = 2, H = 2,
 * D = 64, P = 2: 512 bytes in, 512 bytes out, both inside `buf`) while telling
 * the kernel that its output is one 16-byte vector shorter than it is, so the
 * kernel's own check must refuse the last store: it records
 * H3ATTN_ERR_DEVICE_BOUNDS (tag 5) and skips it.  Every access the kernel
 * makes, refused or not, lies inside `buf`.
 * `buf`: device memory owned by the caller, 16-byte aligned, >= 1024 bytes
 * (contents overwritten).  Asynchronous on `stream`; read the outcome with
 * h3attn_get_device_status().  Returns H3ATTN_ERR_ARG without launching in a
 * build without H3ATTN_BUILD_DEBUG_CHECKS, or for a null, misaligned or too
 * small buffer.
 */
H3ATTN_API int h3attn_selftest_bounds(void* buf, unsigned long long bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* H3ATTN_H */
