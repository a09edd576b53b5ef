/*
 * h3_oracle.c -- plain, slow, fp64 CPU statement of what the attention hot
 * path of a MiniMax-H3-style DiT block computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library: every formula below is written out from its definition.
 *
 * Sources (page title, section):
 *  - QK-RMSNorm: "[feat] Tensor parallelism for MiniMax-H3" (diffusers PR
 *    #14609), PR description: the QK-norms are head_dim-shaped and applied
 *    after the head split.  RMSNorm itself is the textbook definition
 *    y = x / sqrt(mean(x^2) + eps) * w.
 *  - RoPE: same PR description: H3's rotary embedding uses real sin/cos and
 *    broadcasts over the head axis; the loader-bug comment on the same page
 *    shows the angle as the inv_freq buffer times position_ids.  The three
 *    axes (t, h, w) each own a contiguous slice of head_dim.
 *  - Attention: "buqi-minimax-h3-multigpu" README, sections "On accuracy" and
 *    "How it works": every rank evaluates exact full attention over the whole
 *    packed sequence for a subset of the 56 heads.  Softmax(q k^T * scale) v,
 *    restricted to the kv_len valid keys (padding to a multiple of 512, as in
 *    the diffusers PR's NKI comment, contributes nothing).
 *  - Ulysses layout exchange: README "How it works": the sequence stays
 *    row-sharded across P ranks for per-token work, and attention needs every
 *    row for 56/P heads; the all-to-all turns [P][S/P][H][D] into
 *    [P][S][H/P][D] and back.
 *
 * Readings where the pages are silent: eps is an argument (1e-6 in the
 * workloads); rotary pairs are adjacent (2i, 2i+1) inside each axis slice
 * when `interleaved` is 1, or (i, i + d_a/2) when 0; the frequency of pair i
 * in an axis slice of width d_a is theta^(-2i/d_a); scale is 1/sqrt(D) unless
 * given.  Parity against the real H3 checkpoint is not pinned by the pages.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

int h3o_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* RMSNorm over the last axis of a [rows][D] array:
 *   y[r][d] = x[r][d] / sqrt( (1/D) * sum_e x[r][e]^2 + eps ) * w[d]          */
void h3o_rmsnorm(const double *x, const double *w, int64_t rows, int D,
                 double eps, double *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * D;
        double *yr = y + r * D;
        double sum_sq = 0.0;
        for (int d = 0; d < D; ++d)
            sum_sq += xr[d] * xr[d];
        const double rms = sqrt(sum_sq / (double)D + eps);
        for (int d = 0; d < D; ++d)
            yr[d] = xr[d] / rms * w[d];
    }
}

/* Three-axis rotary embedding of a [S][H][D] array.  Axis a in (t, h, w) owns
 * the dims [off_a, off_a + d_a) with off_t = 0, off_h = d_t, off_w = d_t + d_h.
 * Pair i of axis a is rotated by the angle pos[s][a] * theta^(-2i/d_a):
 *   (x0, x1) -> (x0 cos - x1 sin, x0 sin + x1 cos).
 * The same angle is used for every head (the embedding broadcasts over heads). */
void h3o_rope(const double *x, const int32_t *pos, int64_t S, int H, int D,
              int d_t, int d_h, int d_w, double theta, int interleaved,
              double *y)
{
    const int width[3] = { d_t, d_h, d_w };
    const int offset[3] = { 0, d_t, d_t + d_h };
#pragma omp parallel for schedule(static)
    for (int64_t s = 0; s < S; ++s) {
        for (int h = 0; h < H; ++h) {
            const double *xr = x + (s * H + h) * (int64_t)D;
            double *yr = y + (s * H + h) * (int64_t)D;
            for (int d = 0; d < D; ++d)
                yr[d] = xr[d];
            for (int a = 0; a < 3; ++a) {
                const int da = width[a];
                const double p = (double)pos[s * 3 + a];
                for (int i = 0; i < da / 2; ++i) {
                    const double freq = pow(theta, -2.0 * (double)i / (double)da);
                    const double angle = p * freq;
                    const double c = cos(angle), sn = sin(angle);
                    int i0, i1;
                    if (interleaved) {
                        i0 = offset[a] + 2 * i;
                        i1 = offset[a] + 2 * i + 1;
                    } else {
                        i0 = offset[a] + i;
                        i1 = offset[a] + i + da / 2;
                    }
                    yr[i0] = xr[i0] * c - xr[i1] * sn;
                    yr[i1] = xr[i0] * sn + xr[i1] * c;
                }
            }
        }
    }
}

/* Exact softmax attention for every head of a [Sq][H][D] query block against
 * [S][H][D] keys and values, using only keys j < kv_len:
 *   s_j = scale * <q, k_j>,  o = sum_j exp(s_j - max) v_j / sum_j exp(s_j - max).
 * Two passes over the scores (max, then exponentials and sums), all fp64.
 * q rows are independent, so a caller may pass any subset of query rows.    */
void h3o_attention(const double *q, int64_t Sq, const double *k,
                   const double *v, int64_t S, int H, int D, int64_t kv_len,
                   double scale, double *o)
{
    (void)S;
#pragma omp parallel
    {
        double *sc = (double *)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
#pragma omp for schedule(dynamic, 4) collapse(2)
        for (int h = 0; h < H; ++h) {
            for (int64_t r = 0; r < Sq; ++r) {
                const double *qr = q + (r * H + h) * (int64_t)D;
                double *orow = o + (r * H + h) * (int64_t)D;
                double mx = -INFINITY;
                for (int64_t j = 0; j < kv_len; ++j) {
                    const double *kj = k + (j * H + h) * (int64_t)D;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d)
                        dot += qr[d] * kj[d];
                    sc[j] = dot * scale;
                    if (sc[j] > mx)
                        mx = sc[j];
                }
                double denom = 0.0;
                for (int d = 0; d < D; ++d)
                    orow[d] = 0.0;
                for (int64_t j = 0; j < kv_len; ++j) {
                    const double e = exp(sc[j] - mx);
                    const double *vj = v + (j * H + h) * (int64_t)D;
                    denom += e;
                    for (int d = 0; d < D; ++d)
                        orow[d] += e * vj[d];
                }
                for (int d = 0; d < D; ++d)
                    orow[d] /= denom;
            }
        }
        free(sc);
    }
}

/* Ulysses sequence->head exchange, stated per element.  Rank r of P holds the
 * sequence shard in[r][s_local][h][d] (shape [P][S/P][H][D]); after the
 * exchange, rank g holds every row for heads g*H/P .. (g+1)*H/P - 1:
 *   out[g][s][j][d] = in[s / (S/P)][s % (S/P)][g*(H/P) + j][d].
 * Elements are 16-bit words moved unchanged.                                  */
void h3o_seq2head_u16(const uint16_t *in, uint16_t *out, int64_t S, int H,
                      int D, int P)
{
    const int64_t Sp = S / P;
    const int Hp = H / P;
#pragma omp parallel for schedule(static) collapse(2)
    for (int g = 0; g < P; ++g) {
        for (int64_t s = 0; s < S; ++s) {
            const int64_t r = s / Sp, sl = s % Sp;
            for (int j = 0; j < Hp; ++j) {
                for (int d = 0; d < D; ++d) {
                    const int64_t src = ((r * Sp + sl) * H + (g * Hp + j)) * (int64_t)D + d;
                    const int64_t dst = ((g * S + s) * Hp + j) * (int64_t)D + d;
                    out[dst] = in[src];
                }
            }
        }
    }
}

/* Inverse exchange (head->sequence), the output all-to-all:
 *   out[r][s_local][g*(H/P) + j][d] = in[g][r*(S/P) + s_local][j][d].          */
void h3o_head2seq_u16(const uint16_t *in, uint16_t *out, int64_t S, int H,
                      int D, int P)
{
    const int64_t Sp = S / P;
    const int Hp = H / P;
#pragma omp parallel for schedule(static) collapse(2)
    for (int r = 0; r < P; ++r) {
        for (int64_t sl = 0; sl < Sp; ++sl) {
            for (int g = 0; g < P; ++g) {
                for (int j = 0; j < Hp; ++j) {
                    for (int d = 0; d < D; ++d) {
                        const int64_t src = ((g * S + r * Sp + sl) * Hp + j) * (int64_t)D + d;
                        const int64_t dst = ((r * Sp + sl) * H + (g * Hp + j)) * (int64_t)D + d;
                        out[dst] = in[src];
                    }
                }
            }
        }
    }
}

/* ---------------------------------------------------------------------------
 * All-gather exchange variant: the QKV projection through one rank's head
 * rows ("buqi-minimax-h3-multigpu" README, "How it works": for world sizes up
 * to 4 each rank receives the full modulated hidden state and multiplies it by
 * only its own head rows of qkv_proj; slicing the fp8 weight by rows is exact
 * because its scale is one number per tensor).
 *
 * Readings: qkv_proj is a Linear of shape [3*inner, hidden] stored row-major
 * (q rows, then k rows, then v rows; inside each, head h owns rows
 * [h*D, (h+1)*D)); rank r of P owns rows [part*inner + r*inner/P,
 * part*inner + (r+1)*inner/P) of each part; both operands are FP8 E4M3
 * (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
 * S.1111.111 is NaN) with one scale per tensor; no bias term.
 * ------------------------------------------------------------------------- */

/* FP8 E4M3 code -> value, written from the format's definition. */
double h3o_e4m3_decode(uint8_t code)
{
    const int sign = (code >> 7) & 1;
    const int e = (code >> 3) & 0xF;
    const int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);          /* subnormal: 0.m * 2^(1-7) */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);  /* normal: 1.m * 2^(e-7) */
    return sign ? -v : v;
}

/* out[r][part][c] = scale * sum_e x[r][e] * w[part*inner + rank*inner/P + c][e]
 * for the n_rows given rows of x ([n_rows][hidden] codes), part in {q,k,v},
 * c in [0, inner/P).  out is [n_rows][3][inner/P] doubles.                  */
void h3o_qkv_proj_fp8(const uint8_t *x, int64_t n_rows, const uint8_t *w, int hidden, int inner, int P,
                      int rank, double scale, double *out)
{
    const int nr = inner / P;
    double table[256];
    for (int c = 0; c < 256; ++c)
        table[c] = h3o_e4m3_decode((uint8_t)c);
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int64_t r = 0; r < n_rows; ++r) {
        for (int part = 0; part < 3; ++part) {
            const uint8_t *xr = x + r * hidden;
            for (int c = 0; c < nr; ++c) {
                const uint8_t *wr = w + ((int64_t)part * inner + (int64_t)rank * nr + c) * hidden;
                double acc = 0.0;
                for (int e = 0; e < hidden; ++e)
                    acc += table[xr[e]] * table[wr[e]];
                out[(r * 3 + part) * (int64_t)nr + c] = scale * acc;
            }
        }
    }
}
