/*
 * ulysses_oracle.c -- plain CPU oracle for the Ulysses 4D sequence/head relayout.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU baseline leg of the
 * benchmark may load this file's shared library. The product path never calls it and has no CPU
 * fallback. It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes, and where that is stated:
 *
 *   fast-ulysses 0.1.0 (PyPI page), opening paragraph and "Quick start":
 *     one all-to-all trades the sequence shard for a head shard, a second trades it back;
 *     mode 0 maps (b, s_local, n_global, d) -> (b, s_global, n_local, d).
 *   fast-ulysses 0.2.1 (README), "Quick start": mode 1 returns to x's shape.
 *   fast-ulysses 0.1.0, "What it does": per-rank seq_splits / head_splits (uneven shards);
 *     even splits are a special case of the same mapping.
 *   fast-ulysses 0.1.0, "Fusion examples": QK RMSNorm + RoPE inside the scatter.
 *
 * With W ranks, s_q = seq_splits[q], n_r = head_splits[r], S = sum s_q, N = sum n_r,
 * seq_off(q) = sum_{p<q} s_p and head_off(r) = sum_{p<r} n_p, mode 0 is
 *
 *     out[r][bb][seq_off(q) + i][h][j] = in[q][bb][i][head_off(r) + h][j]
 *
 * for every q, r, bb < b, i < s_q, h < n_r, j < d; mode 1 is the same assignment read the
 * other way (out[q][bb][i][head_off(r)+h][j] = in[r][bb][seq_off(q)+i][h][j]). Elements are
 * moved as raw bytes, e bytes each, so the element type never matters.
 *
 * The fused QK transform follows the plainest reading of "QK RMSNorm + RoPE": per head row of
 * d values (bf16 in), RMSNorm over d with eps inside the square root and one weight vector of
 * length d, then rotary embedding on adjacent pairs (2j, 2j+1) with angle p * theta^(-2j/d),
 * where p is the token's global sequence index. Everything is in double; the result is left
 * unrounded (a bf16 round-to-nearest-even helper is provided separately). Its backward (the
 * vector-Jacobian product per row, the output gradient brought back by mode 1) and two variants
 * (fp16 elements; rotate-half pairs (j, j + d/2)) follow at the end of the file.
 *
 * All functions return 0 on success and -1 on invalid arguments.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_MAX_W 8

/* Sum of the first k entries of a split vector: the offset of shard k. */
static int64_t offset_of(const int64_t* splits, int k)
{
    int64_t s = 0;
    for (int p = 0; p < k; ++p) s += splits[p];
    return s;
}

/* Copy one element of e bytes (a constant size per case, so the compiler inlines the copy). */
static void copy_elem(uint8_t* dst, const uint8_t* src, int64_t e)
{
    switch (e) {
        case 1: memcpy(dst, src, 1); break;
        case 2: memcpy(dst, src, 2); break;
        default: memcpy(dst, src, 4); break;
    }
}

static int check_geometry(int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits,
                          int64_t d)
{
    if (W < 1 || W > ORC_MAX_W || b < 1 || d < 1) return -1;
    if (!seq_splits || !head_splits) return -1;
    for (int q = 0; q < W; ++q)
        if (seq_splits[q] < 0 || head_splits[q] < 0) return -1;
    if (offset_of(seq_splits, W) < 1 || offset_of(head_splits, W) < 1) return -1;
    return 0;
}

/*
 * Parts of the fused calls. A whole call walks the source shards q in [0, W) and, in each, the
 * rows i in [0, s_q) of every batch index. The *_part functions below walk only shards
 * q in [q_lo, q_hi) and rows i in [i_lo, min(i_hi, s_q)), in the same order and with the same
 * arithmetic, so that a large check can be split over host threads (the parts write disjoint
 * output rows). The whole-call functions are their part (0, W, 0, INT64_MAX).
 */
static int part_range_ok(int W, int q_lo, int q_hi, int64_t i_lo, int64_t i_hi)
{
    return q_lo >= 0 && q_hi <= W && q_lo <= q_hi && i_lo >= 0 && i_lo <= i_hi ? 0 : -1;
}

static int64_t part_row_end(int64_t s_q, int64_t i_hi) { return i_hi < s_q ? i_hi : s_q; }

/*
 * The relayout, six nested loops, one element (e bytes) per innermost step.
 * in[k] and out[k] are the W ranks' buffers. Mode 0: in[q] is (b, s_q, N, d) and out[r] is
 * (b, S, n_r, d). Mode 1: in[r] is (b, S, n_r, d) and out[q] is (b, s_q, N, d).
 */
int orc_a2a_4d(int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits,
               int64_t d, int64_t e, int mode, const uint8_t* const* in, uint8_t* const* out)
{
    if (check_geometry(W, b, seq_splits, head_splits, d)) return -1;
    if (!(e == 1 || e == 2 || e == 4) || !(mode == 0 || mode == 1)) return -1;
    const int64_t S = offset_of(seq_splits, W);
    const int64_t N = offset_of(head_splits, W);

    for (int q = 0; q < W; ++q) {
        const int64_t s_q = seq_splits[q];
        const int64_t seq_off_q = offset_of(seq_splits, q);
        for (int r = 0; r < W; ++r) {
            const int64_t n_r = head_splits[r];
            const int64_t head_off_r = offset_of(head_splits, r);
            for (int64_t bb = 0; bb < b; ++bb)
                for (int64_t i = 0; i < s_q; ++i)
                    for (int64_t h = 0; h < n_r; ++h)
                        for (int64_t j = 0; j < d; ++j) {
                            /* element index inside rank q's (b, s_q, N, d) tensor */
                            const int64_t seq_side = ((bb * s_q + i) * N + head_off_r + h) * d + j;
                            /* element index inside rank r's (b, S, n_r, d) tensor */
                            const int64_t head_side = ((bb * S + seq_off_q + i) * n_r + h) * d + j;
                            if (mode == 0)
                                copy_elem(out[r] + head_side * e, in[q] + seq_side * e, e);
                            else
                                copy_elem(out[q] + seq_side * e, in[r] + head_side * e, e);
                        }
        }
    }
    return 0;
}

/*
 * Where one output element comes from, read off the same definition: given the output rank and
 * the flat element index inside that rank's output tensor, return the source rank and the flat
 * element index inside that rank's input tensor. Used to check single sampled outputs of
 * workloads too large to relayout on the host.
 */
int orc_a2a_4d_source(int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits,
                      int64_t d, int mode, int out_rank, int64_t out_elem, int* src_rank,
                      int64_t* src_elem)
{
    if (check_geometry(W, b, seq_splits, head_splits, d)) return -1;
    if (!(mode == 0 || mode == 1) || out_rank < 0 || out_rank >= W || out_elem < 0) return -1;
    const int64_t S = offset_of(seq_splits, W);
    const int64_t N = offset_of(head_splits, W);

    if (mode == 0) {
        const int r = out_rank;
        const int64_t n_r = head_splits[r];
        if (out_elem >= b * S * n_r * d) return -1;
        const int64_t j = out_elem % d;
        const int64_t h = (out_elem / d) % n_r;
        const int64_t s = (out_elem / (d * n_r)) % S;
        const int64_t bb = out_elem / (d * n_r * S);
        for (int q = 0; q < W; ++q) {
            const int64_t lo = offset_of(seq_splits, q);
            if (s >= lo && s < lo + seq_splits[q]) {
                const int64_t i = s - lo;
                *src_rank = q;
                *src_elem = ((bb * seq_splits[q] + i) * N + offset_of(head_splits, r) + h) * d + j;
                return 0;
            }
        }
        return -1;
    } else {
        const int q = out_rank;
        const int64_t s_q = seq_splits[q];
        if (out_elem >= b * s_q * N * d) return -1;
        const int64_t j = out_elem % d;
        const int64_t g = (out_elem / d) % N;
        const int64_t i = (out_elem / (d * N)) % s_q;
        const int64_t bb = out_elem / (d * N * s_q);
        for (int r = 0; r < W; ++r) {
            const int64_t lo = offset_of(head_splits, r);
            if (g >= lo && g < lo + head_splits[r]) {
                const int64_t h = g - lo;
                *src_rank = r;
                *src_elem = ((bb * S + offset_of(seq_splits, q) + i) * head_splits[r] + h) * d + j;
                return 0;
            }
        }
        return -1;
    }
}

/* ------------------------------------------------------------------------------------------ */
/* Fused QK RMSNorm + RoPE, in double.                                                         */
/* ------------------------------------------------------------------------------------------ */

/* bf16 bit pattern -> value: bf16 is the upper half of an IEEE binary32. */
double orc_bf16_to_double(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * double -> bf16 bit pattern with one round-to-nearest-even step (8 significand bits, exponent
 * range of binary32, gradual underflow, overflow to infinity).
 */
uint16_t orc_double_to_bf16(double x)
{
    const uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);
    const double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0) return sign;
    int E;
    frexp(a, &E);           /* a in [2^(E-1), 2^E) */
    int ex = E - 1;         /* a in [2^ex, 2^(ex+1)) */
    if (ex < -126) ex = -126; /* below the normal range the spacing stays 2^-133 */
    const double quantum = ldexp(1.0, ex - 7);
    const double k = nearbyint(a / quantum); /* default rounding mode: nearest, ties to even */
    const double v = k * quantum;
    if (v >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u);
    const float f = (float)v; /* exact: v has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

/* RMSNorm over one row of d values: y = x / sqrt(mean(x^2) + eps) * w. */
void orc_rmsnorm(const double* x, int64_t d, const double* w, double eps, double* y)
{
    double sum_sq = 0.0;
    for (int64_t j = 0; j < d; ++j) sum_sq += x[j] * x[j];
    const double mean_sq = sum_sq / (double)d;
    const double inv_rms = 1.0 / sqrt(mean_sq + eps);
    for (int64_t j = 0; j < d; ++j) y[j] = x[j] * inv_rms * w[j];
}

/*
 * Rotary embedding of one row in place, adjacent pairs: for j < d/2 the pair (y[2j], y[2j+1])
 * is rotated by the angle p * theta^(-2j/d).
 */
void orc_rope(double* y, int64_t d, double p, double theta)
{
    for (int64_t j = 0; j < d / 2; ++j) {
        const double freq = pow(theta, -2.0 * (double)j / (double)d);
        const double angle = p * freq;
        const double c = cos(angle), s = sin(angle);
        const double a = y[2 * j], bq = y[2 * j + 1];
        y[2 * j] = a * c - bq * s;
        y[2 * j + 1] = a * s + bq * c;
    }
}

/* One head row: bf16 in -> RMSNorm -> RoPE at position p -> double out. */
static void transform_row(const uint16_t* x_bf16, int64_t d, const double* w, double eps,
                          double p, double theta, double* y)
{
    double* x = (double*)malloc((size_t)d * sizeof(double));
    for (int64_t j = 0; j < d; ++j) x[j] = orc_bf16_to_double(x_bf16[j]);
    orc_rmsnorm(x, d, w, eps, y);
    orc_rope(y, d, p, theta);
    free(x);
}

/*
 * Formulation A: transform each source row where it sits (position p = seq_off(q) + i), then
 * place it where mode 0 puts it. x_in[q] holds rank q's (b, s_q, N, d) bf16 tensor; y_out[r]
 * receives rank r's (b, S, n_r, d) tensor in double.
 */
int orc_qk_fused_A_part(int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits,
                        int64_t d, const uint16_t* const* x_in, const double* w, double eps,
                        double theta, double* const* y_out, int q_lo, int q_hi, int64_t i_lo,
                        int64_t i_hi)
{
    if (check_geometry(W, b, seq_splits, head_splits, d) || (d % 2) != 0) return -1;
    if (part_range_ok(W, q_lo, q_hi, i_lo, i_hi)) return -1;
    const int64_t S = offset_of(seq_splits, W);
    const int64_t N = offset_of(head_splits, W);
    for (int q = q_lo; q < q_hi; ++q) {
        const int64_t s_q = seq_splits[q];
        const int64_t seq_off_q = offset_of(seq_splits, q);
        for (int64_t bb = 0; bb < b; ++bb)
            for (int64_t i = i_lo; i < part_row_end(s_q, i_hi); ++i)
                for (int64_t g = 0; g < N; ++g) {
                    /* the destination rank owns global head g */
                    int r = 0;
                    while (!(g >= offset_of(head_splits, r) &&
                             g < offset_of(head_splits, r) + head_splits[r]))
                        ++r;
                    const int64_t n_r = head_splits[r];
                    const int64_t h = g - offset_of(head_splits, r);
                    const uint16_t* src = x_in[q] + ((bb * s_q + i) * N + g) * d;
                    double* dst = y_out[r] + ((bb * S + seq_off_q + i) * n_r + h) * d;
                    transform_row(src, d, w, eps, (double)(seq_off_q + i), theta, dst);
                }
    }
    return 0;
}

int orc_qk_fused_A(int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits,
                   int64_t d, const uint16_t* const* x_in, const double* w, double eps,
                   double theta, double* const* y_out)
{
    return orc_qk_fused_A_part(W, b, seq_splits, head_splits, d, x_in, w, eps, theta, y_out, 0, W,
                               0, INT64_MAX);
}

/*
 * Formulation B: relayout the bf16 bytes first (mode 0), then transform each destination row
 * with p = its index along the output's global sequence axis.
 */
int orc_qk_fused_B(int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits,
                   int64_t d, const uint16_t* const* x_in, const double* w, double eps,
                   double theta, double* const* y_out)
{
    if (check_geometry(W, b, seq_splits, head_splits, d) || (d % 2) != 0) return -1;
    const int64_t S = offset_of(seq_splits, W);
    uint8_t* moved[ORC_MAX_W] = {0};
    for (int r = 0; r < W; ++r)
        moved[r] = (uint8_t*)malloc((size_t)(b * S * head_splits[r] * d * 2 + 1));
    int rc = orc_a2a_4d(W, b, seq_splits, head_splits, d, 2, 0, (const uint8_t* const*)x_in,
                        moved);
    if (rc == 0) {
        for (int r = 0; r < W; ++r) {
            const int64_t n_r = head_splits[r];
            for (int64_t bb = 0; bb < b; ++bb)
                for (int64_t s = 0; s < S; ++s)
                    for (int64_t h = 0; h < n_r; ++h) {
                        const int64_t row = (bb * S + s) * n_r + h;
                        transform_row((const uint16_t*)moved[r] + row * d, d, w, eps, (double)s,
                                      theta, y_out[r] + row * d);
                    }
        }
    }
    for (int r = 0; r < W; ++r) free(moved[r]);
    return rc;
}

/*
 * One output row of the fused transform, for sampled checks of large workloads: rank r's row
 * (bb, s, h) of its (b, S, n_r, d) output, computed from the source row the definition names.
 */
int orc_qk_fused_row(int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits,
                     int64_t d, int r, int64_t bb, int64_t s, int64_t h,
                     const uint16_t* const* x_in, const double* w, double eps, double theta,
                     double* y)
{
    if (check_geometry(W, b, seq_splits, head_splits, d) || (d % 2) != 0) return -1;
    if (r < 0 || r >= W || bb < 0 || bb >= b || h < 0 || h >= head_splits[r]) return -1;
    if (s < 0 || s >= offset_of(seq_splits, W)) return -1;
    const int64_t N = offset_of(head_splits, W);
    for (int q = 0; q < W; ++q) {
        const int64_t lo = offset_of(seq_splits, q);
        if (s >= lo && s < lo + seq_splits[q]) {
            const int64_t i = s - lo;
            const uint16_t* src =
                x_in[q] + ((bb * seq_splits[q] + i) * N + offset_of(head_splits, r) + h) * d;
            transform_row(src, d, w, eps, (double)s, theta, y);
            return 0;
        }
    }
    return -1;
}

/* Element-wise array forms of the two bf16 conversions above. */
void orc_bf16_to_double_array(const uint16_t* h, int64_t n, double* out)
{
    for (int64_t k = 0; k < n; ++k) out[k] = orc_bf16_to_double(h[k]);
}

void orc_double_to_bf16_array(const double* x, int64_t n, uint16_t* out)
{
    for (int64_t k = 0; k < n; ++k) out[k] = orc_double_to_bf16(x[k]);
}

/*
 * Interleaved packed QKV, the layout a fused QKV projection writes (FastVideo, "Ulysses
 * performance on GB200": packed QKV): rank q holds one (b, s_q, 3, N, d) bf16 tensor whose plane 0
 * is q, plane 1 is k and plane 2 is v. q and k rows are transformed as orc_qk_fused_A does (with
 * wq and wk respectively) and placed where mode 0 puts them (double outputs); v rows are placed by
 * mode 0 unchanged (bf16 bit patterns). q_out[r], k_out[r], v_out[r] are rank r's (b, S, n_r, d).
 */
int orc_qkv_fused_part(int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits,
                       int64_t d, const uint16_t* const* qkv_in, const double* wq,
                       const double* wk, double eps, double theta, double* const* q_out,
                       double* const* k_out, uint16_t* const* v_out, int q_lo, int q_hi,
                       int64_t i_lo, int64_t i_hi)
{
    if (check_geometry(W, b, seq_splits, head_splits, d) || (d % 2) != 0) return -1;
    if (part_range_ok(W, q_lo, q_hi, i_lo, i_hi)) return -1;
    const int64_t S = offset_of(seq_splits, W);
    const int64_t N = offset_of(head_splits, W);
    for (int q = q_lo; q < q_hi; ++q) {
        const int64_t s_q = seq_splits[q];
        const int64_t seq_off_q = offset_of(seq_splits, q);
        for (int64_t bb = 0; bb < b; ++bb)
            for (int64_t i = i_lo; i < part_row_end(s_q, i_hi); ++i)
                for (int64_t g = 0; g < N; ++g) {
                    int r = 0;
                    while (!(g >= offset_of(head_splits, r) &&
                             g < offset_of(head_splits, r) + head_splits[r]))
                        ++r;
                    const int64_t n_r = head_splits[r];
                    const int64_t h = g - offset_of(head_splits, r);
                    const int64_t dst_row = ((bb * S + seq_off_q + i) * n_r + h) * d;
                    const double p = (double)(seq_off_q + i);
                    /* row (bb, i, plane, g) of rank q's (b, s_q, 3, N, d) tensor */
                    const uint16_t* qrow = qkv_in[q] + (((bb * s_q + i) * 3 + 0) * N + g) * d;
                    const uint16_t* krow = qkv_in[q] + (((bb * s_q + i) * 3 + 1) * N + g) * d;
                    const uint16_t* vrow = qkv_in[q] + (((bb * s_q + i) * 3 + 2) * N + g) * d;
                    transform_row(qrow, d, wq, eps, p, theta, q_out[r] + dst_row);
                    transform_row(krow, d, wk, eps, p, theta, k_out[r] + dst_row);
                    for (int64_t j = 0; j < d; ++j) v_out[r][dst_row + j] = vrow[j];
                }
    }
    return 0;
}

int orc_qkv_fused(int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits,
                  int64_t d, const uint16_t* const* qkv_in, const double* wq, const double* wk,
                  double eps, double theta, double* const* q_out, double* const* k_out,
                  uint16_t* const* v_out)
{
    return orc_qkv_fused_part(W, b, seq_splits, head_splits, d, qkv_in, wq, wk, eps, theta, q_out,
                              k_out, v_out, 0, W, 0, INT64_MAX);
}

/*
 * Packed inputs with C planes per token, the general form of the interleaved layout (FastVideo,
 * "Ulysses performance on GB200": packed QKV or QKVG). Rank q's input holds b * s_q tokens; token
 * (bb, i) starts (bb * s_q + i) * pitch elements into it (pitch >= C * N * d: a token may carry
 * further columns, which are never read), and within a token plane c's head g is the d elements at
 * c * N * d + g * d. Planes q_plane and k_plane are transformed as orc_qk_fused_A does (with wq and
 * wk) and placed where mode 0 puts them (double, q_out[r] and k_out[r]); every other plane c is
 * placed by mode 0 unchanged (bf16 bit patterns, plain_out[c * W + r]; the entries of the q and k
 * planes are not touched). Every output is rank r's (b, S, n_r, d).
 */
int orc_packed_fused(int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits,
                     int64_t d, int planes, int q_plane, int k_plane, int64_t pitch,
                     const uint16_t* const* in, const double* wq, const double* wk, double eps,
                     double theta, double* const* q_out, double* const* k_out,
                     uint16_t* const* plain_out)
{
    if (check_geometry(W, b, seq_splits, head_splits, d) || (d % 2) != 0) return -1;
    const int64_t S = offset_of(seq_splits, W);
    const int64_t N = offset_of(head_splits, W);
    if (planes < 2 || q_plane < 0 || q_plane >= planes || k_plane < 0 || k_plane >= planes ||
        q_plane == k_plane || pitch < planes * N * d)
        return -1;
    for (int q = 0; q < W; ++q) {
        const int64_t s_q = seq_splits[q];
        const int64_t seq_off_q = offset_of(seq_splits, q);
        for (int64_t bb = 0; bb < b; ++bb)
            for (int64_t i = 0; i < s_q; ++i) {
                const uint16_t* token = in[q] + (bb * s_q + i) * pitch;
                const double p = (double)(seq_off_q + i);
                for (int c = 0; c < planes; ++c)
                    for (int64_t g = 0; g < N; ++g) {
                        int r = 0;
                        while (!(g >= offset_of(head_splits, r) &&
                                 g < offset_of(head_splits, r) + head_splits[r]))
                            ++r;
                        const int64_t n_r = head_splits[r];
                        const int64_t h = g - offset_of(head_splits, r);
                        const int64_t dst_row = ((bb * S + seq_off_q + i) * n_r + h) * d;
                        const uint16_t* row = token + (c * N + g) * d;
                        if (c == q_plane)
                            transform_row(row, d, wq, eps, p, theta, q_out[r] + dst_row);
                        else if (c == k_plane)
                            transform_row(row, d, wk, eps, p, theta, k_out[r] + dst_row);
                        else
                            for (int64_t j = 0; j < d; ++j) plain_out[c * W + r][dst_row + j] = row[j];
                    }
            }
    }
    return 0;
}

/*
 * Backward of the fused transform for one row (vector-Jacobian product). The forward row is
 * y = R(p) (x * w / rms(x)) with rms(x) = sqrt(mean(x^2) + eps) and R(p) the rotation above.
 * Given g = dL/dy: u = R(-p) g (the rotation is orthogonal), a = u * w,
 * dL/dx = (a - xh * mean(a * xh)) / rms(x) with xh = x / rms(x), and dL/dw += u * xh.
 * row_bwd_core is the RMSNorm part, given u; orc_fused_row_bwd rotates g back first.
 */
static void row_bwd_core(const double* x, const double* u, int64_t d, const double* w, double eps,
                         double* dx, double* dw_acc)
{
    double sum_sq = 0.0;
    for (int64_t j = 0; j < d; ++j) sum_sq += x[j] * x[j];
    const double inv_rms = 1.0 / sqrt(sum_sq / (double)d + eps);
    double dot = 0.0;
    for (int64_t j = 0; j < d; ++j) {
        const double xh = x[j] * inv_rms;
        dot += u[j] * w[j] * xh;
        dw_acc[j] += u[j] * xh;
    }
    for (int64_t j = 0; j < d; ++j) {
        const double xh = x[j] * inv_rms;
        dx[j] = inv_rms * (u[j] * w[j] - xh * dot / (double)d);
    }
}

void orc_fused_row_bwd(const double* x, const double* g, int64_t d, const double* w, double eps,
                       double p, double theta, double* dx, double* dw_acc)
{
    double* u = (double*)malloc((size_t)d * sizeof(double));
    for (int64_t j = 0; j < d; ++j) u[j] = g[j];
    orc_rope(u, d, -p, theta);
    row_bwd_core(x, u, d, w, eps, dx, dw_acc);
    free(u);
}

/*
 * Backward of the fused mode-0 call for one tensor: x_in[q] is rank q's forward input
 * (b, s_q, N, d) bf16, g_out[r] rank r's gradient with respect to the forward output
 * (b, S, n_r, d) bf16. dx[q] receives rank q's gradient with respect to its input (double,
 * (b, s_q, N, d)); dw (d values) is set to the gradient with respect to the weight (for a part,
 * to the sum over that part's rows).
 */
int orc_qk_fused_bwd_part(int W, int64_t b, const int64_t* seq_splits,
                          const int64_t* head_splits, int64_t d, const uint16_t* const* x_in,
                          const uint16_t* const* g_out, const double* w, double eps, double theta,
                          double* const* dx, double* dw, int q_lo, int q_hi, int64_t i_lo,
                          int64_t i_hi)
{
    if (check_geometry(W, b, seq_splits, head_splits, d) || (d % 2) != 0) return -1;
    if (part_range_ok(W, q_lo, q_hi, i_lo, i_hi)) return -1;
    const int64_t S = offset_of(seq_splits, W);
    const int64_t N = offset_of(head_splits, W);
    double* x = (double*)malloc((size_t)d * sizeof(double));
    double* g = (double*)malloc((size_t)d * sizeof(double));
    for (int64_t j = 0; j < d; ++j) dw[j] = 0.0;
    for (int q = q_lo; q < q_hi; ++q) {
        const int64_t s_q = seq_splits[q];
        const int64_t seq_off_q = offset_of(seq_splits, q);
        for (int64_t bb = 0; bb < b; ++bb)
            for (int64_t i = i_lo; i < part_row_end(s_q, i_hi); ++i)
                for (int64_t hg = 0; hg < N; ++hg) {
                    int r = 0;
                    while (!(hg >= offset_of(head_splits, r) &&
                             hg < offset_of(head_splits, r) + head_splits[r]))
                        ++r;
                    const int64_t n_r = head_splits[r];
                    const int64_t h = hg - offset_of(head_splits, r);
                    const int64_t src_row = ((bb * s_q + i) * N + hg) * d;
                    const int64_t out_row = ((bb * S + seq_off_q + i) * n_r + h) * d;
                    for (int64_t j = 0; j < d; ++j) {
                        x[j] = orc_bf16_to_double(x_in[q][src_row + j]);
                        g[j] = orc_bf16_to_double(g_out[r][out_row + j]);
                    }
                    orc_fused_row_bwd(x, g, d, w, eps, (double)(seq_off_q + i), theta,
                                      dx[q] + src_row, dw);
                }
    }
    free(x);
    free(g);
    return 0;
}

int orc_qk_fused_bwd(int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits,
                     int64_t d, const uint16_t* const* x_in, const uint16_t* const* g_out,
                     const double* w, double eps, double theta, double* const* dx, double* dw)
{
    return orc_qk_fused_bwd_part(W, b, seq_splits, head_splits, d, x_in, g_out, w, eps, theta, dx,
                                 dw, 0, W, 0, INT64_MAX);
}

/*
 * Backward of orc_packed_fused (same packing and planes): packed_in holds the forward's packed
 * inputs (only the q and k planes are read), grads[c * W + r] rank r's gradient of plane c's
 * output ((b, S, n_r, d) bf16). Written into dpacked (rank q's packed layout, the same pitch):
 * for the q and k planes the gradient of their rows through the fused transform (double, as
 * orc_qk_fused_bwd computes it, with wq and wk), for every other plane its gradient brought back
 * by mode 1 (the bf16 bit patterns, widened exactly to double); the columns of a token beyond its
 * planes are not touched. dw[0 .. d) and dw[d .. 2d) are set to the gradients of wq and wk.
 */
int orc_packed_fused_bwd(int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits,
                         int64_t d, int planes, int q_plane, int k_plane, int64_t pitch,
                         const uint16_t* const* packed_in, const uint16_t* const* grads,
                         const double* wq, const double* wk, double eps, double theta,
                         double* const* dpacked, double* dw)
{
    if (check_geometry(W, b, seq_splits, head_splits, d) || (d % 2) != 0) return -1;
    const int64_t S = offset_of(seq_splits, W);
    const int64_t N = offset_of(head_splits, W);
    if (planes < 2 || q_plane < 0 || q_plane >= planes || k_plane < 0 || k_plane >= planes ||
        q_plane == k_plane || pitch < planes * N * d)
        return -1;
    double* x = (double*)malloc((size_t)d * sizeof(double));
    double* g = (double*)malloc((size_t)d * sizeof(double));
    for (int64_t j = 0; j < 2 * d; ++j) dw[j] = 0.0;
    for (int q = 0; q < W; ++q) {
        const int64_t s_q = seq_splits[q];
        const int64_t seq_off_q = offset_of(seq_splits, q);
        for (int64_t bb = 0; bb < b; ++bb)
            for (int64_t i = 0; i < s_q; ++i) {
                const int64_t token = (bb * s_q + i) * pitch;
                for (int c = 0; c < planes; ++c)
                    for (int64_t hg = 0; hg < N; ++hg) {
                        int r = 0;
                        while (!(hg >= offset_of(head_splits, r) &&
                                 hg < offset_of(head_splits, r) + head_splits[r]))
                            ++r;
                        const int64_t n_r = head_splits[r];
                        const int64_t h = hg - offset_of(head_splits, r);
                        const int64_t at = token + (c * N + hg) * d;
                        const int64_t head_row = ((bb * S + seq_off_q + i) * n_r + h) * d;
                        const uint16_t* gr = grads[c * W + r] + head_row;
                        if (c == q_plane || c == k_plane) {
                            for (int64_t j = 0; j < d; ++j) {
                                x[j] = orc_bf16_to_double(packed_in[q][at + j]);
                                g[j] = orc_bf16_to_double(gr[j]);
                            }
                            orc_fused_row_bwd(x, g, d, c == q_plane ? wq : wk, eps,
                                              (double)(seq_off_q + i), theta, dpacked[q] + at,
                                              c == q_plane ? dw : dw + d);
                        } else {
                            for (int64_t j = 0; j < d; ++j)
                                dpacked[q][at + j] = orc_bf16_to_double(gr[j]);
                        }
                    }
            }
    }
    free(x);
    free(g);
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Variants of the fused call: fp16 elements and rotate-half RoPE pairs.                        */
/* ------------------------------------------------------------------------------------------ */
/*
 * The pages list float16 among the element types (fast-ulysses 0.2.1, "Limits") and name the
 * fused QK RMSNorm + RoPE without fixing its pair layout. Besides adjacent pairs (2j, 2j+1), the
 * other common layout ("rotate half") pairs element j with element j + d/2; both use the angle
 * p * theta^(-2j/d) for pair j. Functions below take f16 (0: bf16 elements, 1: IEEE binary16)
 * and half_pairs (0: adjacent, 1: rotate half).
 */

/* binary16 bit pattern -> value (exact): 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double orc_f16_to_double(uint16_t h)
{
    const int negative = (h >> 15) & 1;
    const int field = (h >> 10) & 0x1F;
    const int fraction = h & 0x3FF;
    double v;
    if (field == 0)
        v = ldexp((double)fraction, -24);                /* zero or subnormal: fraction * 2^-24 */
    else if (field == 31)
        v = fraction ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + fraction), field - 25); /* (1.fraction) * 2^(field - 15) */
    return negative ? -v : v;
}

/*
 * double -> binary16 bit pattern with one round-to-nearest-even step (11 significand bits,
 * normal exponents down to -14, gradual underflow in steps of 2^-24, overflow to infinity).
 */
uint16_t orc_double_to_f16(double x)
{
    const uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7E00u);
    const double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7C00u);
    if (a == 0.0) return sign;
    int E;
    frexp(a, &E);
    int ex = E - 1;           /* a in [2^ex, 2^(ex+1)) */
    if (ex < -14) ex = -14;   /* below the normal range the spacing stays 2^-24 */
    const double step = ldexp(1.0, ex - 10);
    const double v = nearbyint(a / step) * step; /* default rounding mode: nearest, ties to even */
    if (v >= 65536.0) return (uint16_t)(sign | 0x7C00u); /* 65520 and up round past 65504 */
    if (v == 0.0) return sign;                             /* below 2^-25: rounds to zero */
    int Ev;
    frexp(v, &Ev);
    const int ev = Ev - 1;
    if (ev < -14) return (uint16_t)(sign | (uint16_t)(v / ldexp(1.0, -24))); /* subnormal */
    const uint16_t frac = (uint16_t)(v / ldexp(1.0, ev - 10) - 1024.0);
    return (uint16_t)(sign | (uint16_t)((ev + 15) << 10) | frac);
}

void orc_f16_to_double_array(const uint16_t* h, int64_t n, double* out)
{
    for (int64_t k = 0; k < n; ++k) out[k] = orc_f16_to_double(h[k]);
}

void orc_double_to_f16_array(const double* x, int64_t n, uint16_t* out)
{
    for (int64_t k = 0; k < n; ++k) out[k] = orc_double_to_f16(x[k]);
}

/*
 * Rotary embedding of one row in place, rotate-half pairs: for j < d/2 the pair
 * (y[j], y[j + d/2]) is rotated by the angle p * theta^(-2j/d).
 */
void orc_rope_half(double* y, int64_t d, double p, double theta)
{
    const int64_t half = d / 2;
    for (int64_t j = 0; j < half; ++j) {
        const double angle = p * pow(theta, -(double)(2 * j) / (double)d);
        const double c = cos(angle), s = sin(angle);
        const double first = y[j], second = y[half + j];
        y[j] = first * c - second * s;
        y[half + j] = first * s + second * c;
    }
}

static double decode_elem(uint16_t h, int f16)
{
    return f16 ? orc_f16_to_double(h) : orc_bf16_to_double(h);
}

static void rope_pairs(double* y, int64_t d, double p, double theta, int half_pairs)
{
    if (half_pairs)
        orc_rope_half(y, d, p, theta);
    else
        orc_rope(y, d, p, theta);
}

/* One head row of a variant: decode, RMSNorm, RoPE at position p; double out. */
void orc_fused_row_var(const uint16_t* x_raw, int64_t d, int f16, int half_pairs, const double* w,
                       double eps, double p, double theta, double* y)
{
    double* x = (double*)malloc((size_t)d * sizeof(double));
    for (int64_t j = 0; j < d; ++j) x[j] = decode_elem(x_raw[j], f16);
    orc_rmsnorm(x, d, w, eps, y);
    rope_pairs(y, d, p, theta, half_pairs);
    free(x);
}

/*
 * The fused mode-0 call of a variant for one tensor: every source row is transformed at its
 * global position seq_off(q) + i and placed where mode 0 puts it. x_in[q]: rank q's
 * (b, s_q, N, d) elements; y_out[r]: rank r's (b, S, n_r, d) in double.
 */
int orc_qk_fused_var_part(int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits,
                          int64_t d, int f16, int half_pairs, const uint16_t* const* x_in,
                          const double* w, double eps, double theta, double* const* y_out,
                          int q_lo, int q_hi, int64_t i_lo, int64_t i_hi)
{
    if (check_geometry(W, b, seq_splits, head_splits, d) || (d % 2) != 0) return -1;
    if (part_range_ok(W, q_lo, q_hi, i_lo, i_hi)) return -1;
    const int64_t S = offset_of(seq_splits, W);
    const int64_t N = offset_of(head_splits, W);
    for (int r = 0; r < W; ++r) {
        const int64_t n_r = head_splits[r];
        const int64_t first_head = offset_of(head_splits, r);
        for (int q = q_lo; q < q_hi; ++q) {
            const int64_t s_q = seq_splits[q];
            const int64_t seq_off_q = offset_of(seq_splits, q);
            for (int64_t bb = 0; bb < b; ++bb)
                for (int64_t i = i_lo; i < part_row_end(s_q, i_hi); ++i)
                    for (int64_t h = 0; h < n_r; ++h) {
                        const uint16_t* src = x_in[q] + ((bb * s_q + i) * N + first_head + h) * d;
                        double* dst = y_out[r] + ((bb * S + seq_off_q + i) * n_r + h) * d;
                        orc_fused_row_var(src, d, f16, half_pairs, w, eps,
                                          (double)(seq_off_q + i), theta, dst);
                    }
        }
    }
    return 0;
}

int orc_qk_fused_var(int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits,
                     int64_t d, int f16, int half_pairs, const uint16_t* const* x_in,
                     const double* w, double eps, double theta, double* const* y_out)
{
    return orc_qk_fused_var_part(W, b, seq_splits, head_splits, d, f16, half_pairs, x_in, w, eps,
                                 theta, y_out, 0, W, 0, INT64_MAX);
}

/* Row backward of a variant: g rotated back with the variant's pairs, then the RMSNorm part. */
void orc_fused_row_bwd_var(const double* x, const double* g, int64_t d, int half_pairs,
                           const double* w, double eps, double p, double theta, double* dx,
                           double* dw_acc)
{
    double* u = (double*)malloc((size_t)d * sizeof(double));
    for (int64_t j = 0; j < d; ++j) u[j] = g[j];
    rope_pairs(u, d, -p, theta, half_pairs);
    row_bwd_core(x, u, d, w, eps, dx, dw_acc);
    free(u);
}

/*
 * Backward of a variant's fused call for one tensor: x_in[q] rank q's forward input
 * (b, s_q, N, d), g_out[r] rank r's output gradient (b, S, n_r, d), both in the variant's
 * element type; dx[q] (double, (b, s_q, N, d)) and dw (d values, cleared first) as
 * orc_qk_fused_bwd (for a part, dw is the sum over that part's rows).
 */
int orc_qk_fused_bwd_var_part(int W, int64_t b, const int64_t* seq_splits,
                              const int64_t* head_splits, int64_t d, int f16, int half_pairs,
                              const uint16_t* const* x_in, const uint16_t* const* g_out,
                              const double* w, double eps, double theta, double* const* dx,
                              double* dw, int q_lo, int q_hi, int64_t i_lo, int64_t i_hi)
{
    if (check_geometry(W, b, seq_splits, head_splits, d) || (d % 2) != 0) return -1;
    if (part_range_ok(W, q_lo, q_hi, i_lo, i_hi)) return -1;
    const int64_t S = offset_of(seq_splits, W);
    const int64_t N = offset_of(head_splits, W);
    double* x = (double*)malloc((size_t)d * sizeof(double));
    double* g = (double*)malloc((size_t)d * sizeof(double));
    memset(dw, 0, (size_t)d * sizeof(double));
    for (int r = 0; r < W; ++r) {
        const int64_t n_r = head_splits[r];
        const int64_t first_head = offset_of(head_splits, r);
        for (int q = q_lo; q < q_hi; ++q) {
            const int64_t s_q = seq_splits[q];
            const int64_t seq_off_q = offset_of(seq_splits, q);
            for (int64_t bb = 0; bb < b; ++bb)
                for (int64_t i = i_lo; i < part_row_end(s_q, i_hi); ++i)
                    for (int64_t h = 0; h < n_r; ++h) {
                        const int64_t in_row = ((bb * s_q + i) * N + first_head + h) * d;
                        const int64_t grad_row = ((bb * S + seq_off_q + i) * n_r + h) * d;
                        for (int64_t j = 0; j < d; ++j) {
                            x[j] = decode_elem(x_in[q][in_row + j], f16);
                            g[j] = decode_elem(g_out[r][grad_row + j], f16);
                        }
                        orc_fused_row_bwd_var(x, g, d, half_pairs, w, eps,
                                              (double)(seq_off_q + i), theta, dx[q] + in_row, dw);
                    }
        }
    }
    free(x);
    free(g);
    return 0;
}

int orc_qk_fused_bwd_var(int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits,
                         int64_t d, int f16, int half_pairs, const uint16_t* const* x_in,
                         const uint16_t* const* g_out, const double* w, double eps, double theta,
                         double* const* dx, double* dw)
{
    return orc_qk_fused_bwd_var_part(W, b, seq_splits, head_splits, d, f16, half_pairs, x_in,
                                     g_out, w, eps, theta, dx, dw, 0, W, 0, INT64_MAX);
}
