// plan.cpp -- the host-side addressing plan: validation, prefix sums, chunking along the sequence
// shards, and the work-unit tables handed to the kernels by value. Makes no CUDA call, so it can
// be tested without a GPU (fast-ulysses 0.1.0, "What it does": the addressing is a host-side
// plan, testable without a GPU).
#include "plan.h"

#include <algorithm>
#include <cmath>
#include <cstring>

#include "../../include/ulysses.h"

namespace uly {

int64_t elem_size_of(int dtype)
{
    switch (dtype) {
        case ULY_U8:
        case ULY_F8E4M3:
        case ULY_F8E5M2:
        case ULY_I8: return 1;
        case ULY_F16:
        case ULY_BF16: return 2;
        case ULY_F32: return 4;
        default: return 0;
    }
}

static bool mul_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_mul_overflow(a, b, out); }

int plan_init(Plan* p, int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits,
              int64_t d, int dtype)
{
    if (!p || !seq_splits || !head_splits) return ULY_EINVAL;
    if (W < 1 || W > kMaxW || b < 1 || d < 1) return ULY_EINVAL;
    const int64_t e = elem_size_of(dtype);
    if (e == 0) return ULY_EINVAL;
    std::memset(p, 0, sizeof *p);
    p->W = W;
    p->dtype = dtype;
    p->b = b;
    p->d = d;
    p->e = e;
    int64_t S = 0, N = 0;
    for (int k = 0; k < W; ++k) {
        if (seq_splits[k] < 0 || head_splits[k] < 0) return ULY_EINVAL;
        p->s[k] = seq_splits[k];
        p->n[k] = head_splits[k];
        p->seq_off[k] = S;
        p->head_off[k] = N;
        if (__builtin_add_overflow(S, seq_splits[k], &S)) return ULY_EINVAL;
        if (__builtin_add_overflow(N, head_splits[k], &N)) return ULY_EINVAL;
    }
    p->seq_off[W] = S;
    p->head_off[W] = N;
    if (S < 1 || N < 1) return ULY_EINVAL;
    p->S = S;
    p->N = N;
    // every byte offset the kernels form must fit in int64 with room to spare
    int64_t t;
    if (!mul_ok(b, S, &t) || !mul_ok(t, N, &t) || !mul_ok(t, d, &t) || !mul_ok(t, e, &t) ||
        t > (int64_t(1) << 60))
        return ULY_EINVAL;
    if ((d * e) % 16 != 0) return ULY_EALIGN;
    p->chunk_cap = int64_t(1) << 30;
    p->max_ctas = 0;
    p->rope_half = 0;
    p->fused_engine = 0;
    return ULY_OK;
}

int64_t seq_side_bytes(const Plan& p, int q) { return p.b * p.s[q] * p.N * p.d * p.e; }
int64_t head_side_bytes(const Plan& p, int r) { return p.b * p.S * p.n[r] * p.d * p.e; }

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Largest per-rank byte count of any launch when the shards are cut into C chunks, bounded
// through ceil(s_q / C) rows per shard (which is monotone in C).
static bool chunking_fits(const Plan& p, int64_t C)
{
    const int64_t row = p.d * p.e;
    int64_t rows_all = 0;
    for (int q = 0; q < p.W; ++q) {
        const int64_t rq = ceil_div(p.s[q], C);
        rows_all += rq;
        if (p.b * rq * p.N * row > p.chunk_cap) return false;  // rank q's seq-side tensor
    }
    for (int r = 0; r < p.W; ++r)
        if (p.b * rows_all * p.n[r] * row > p.chunk_cap) return false;  // rank r's head side
    return true;
}

int num_chunks(const Plan& p, int64_t* n_chunks)
{
    int64_t hi = 1;
    for (int q = 0; q < p.W; ++q) hi = p.s[q] > hi ? p.s[q] : hi;
    if (!chunking_fits(p, hi)) return ULY_ECHUNK;
    int64_t lo = 1;
    while (lo < hi) {  // smallest C in [lo, hi] that fits
        const int64_t mid = lo + (hi - lo) / 2;
        if (chunking_fits(p, mid))
            hi = mid;
        else
            lo = mid + 1;
    }
    *n_chunks = lo;
    return ULY_OK;
}

void chunk_rows(const Plan& p, int64_t C, int64_t c, ChunkRows* out)
{
    std::memset(out, 0, sizeof *out);
    for (int q = 0; q < p.W; ++q) {
        const __int128 s = p.s[q];
        const int64_t lo = int64_t(s * c / C);
        const int64_t hi = int64_t(s * (c + 1) / C);
        out->lo[q] = lo;
        out->cnt[q] = hi - lo;
    }
}

void global_chunk_rows(const Plan& p, int64_t lo, int64_t hi, ChunkRows* out)
{
    std::memset(out, 0, sizeof *out);
    for (int q = 0; q < p.W; ++q) {
        const int64_t a = std::min(std::max(lo - p.seq_off[q], int64_t(0)), p.s[q]);
        const int64_t b = std::min(std::max(hi - p.seq_off[q], int64_t(0)), p.s[q]);
        out->lo[q] = a;
        out->cnt[q] = b - a;
    }
}

int64_t global_chunk_span(const Plan& p, int64_t target_chunks)
{
    const int64_t seq_row = p.b * p.N * p.d * p.e;  // one global row, all ranks' heads, all batches
    if (seq_row > p.chunk_cap) return 0;
    int64_t span = (p.S + target_chunks - 1) / target_chunks;
    const int64_t cap_rows = p.chunk_cap / seq_row;
    return span < cap_rows ? (span > 0 ? span : 1) : cap_rows;
}

void build_relayout_units(const Plan& p, const ChunkRows& rows, int64_t unit_bytes, RelayoutArgs* a)
{
    const int W = p.W;
    a->W = W;
    a->unit_bytes = int32_t(unit_bytes);
    a->S = p.S;
    a->N = p.N;
    a->b = p.b;
    a->d_bytes = p.d * p.e;
    for (int k = 0; k < kMaxW; ++k) {
        const bool live = k < W;
        a->s[k] = live ? p.s[k] : 0;
        a->seq_off[k] = live ? p.seq_off[k] : 0;
        a->n[k] = live ? p.n[k] : 0;
        a->head_off[k] = live ? p.head_off[k] : 0;
        a->row_lo[k] = live ? rows.lo[k] : 0;
        a->rows[k] = live ? rows.cnt[k] : 0;
        const int64_t run = a->n[k] * a->d_bytes;
        if (run == 0) {
            a->rows_per_unit[k] = 1;
            a->pieces[k] = 1;
        } else if (run <= unit_bytes) {
            a->rows_per_unit[k] = unit_bytes / run;
            a->pieces[k] = 1;
        } else {
            a->rows_per_unit[k] = 1;
            a->pieces[k] = ceil_div(run, unit_bytes);
        }
    }
    int64_t total = 0;
    for (int g = 0; g <= kMaxSeg; ++g) {
        a->unit_begin[g] = total;
        if (g == kMaxSeg || g >= W * W) continue;
        const int q = g / W, r = g % W;
        if (a->rows[q] == 0 || a->n[r] == 0) continue;
        total += p.b * ceil_div(a->rows[q], a->rows_per_unit[r]) * a->pieces[r];
    }
    a->total_units = total;
}

void build_row_tiles(const Plan& p, const ChunkRows& rows, int64_t tile_rows, RowTileArgs* a)
{
    const int W = p.W;
    a->W = W;
    a->S = p.S;
    a->N = p.N;
    a->b = p.b;
    a->d_bytes = p.d * p.e;
    a->tile_rows = tile_rows;
    int64_t total = 0;
    for (int k = 0; k < kMaxW; ++k) {
        const bool live = k < W;
        a->s[k] = live ? p.s[k] : 0;
        a->seq_off[k] = live ? p.seq_off[k] : 0;
        a->n[k] = live ? p.n[k] : 0;
        a->head_off[k] = live ? p.head_off[k] : 0;
        a->row_lo[k] = live ? rows.lo[k] : 0;
        a->rows[k] = live ? rows.cnt[k] : 0;
        a->unit_begin[k] = total;
        if (live) total += p.b * ceil_div(a->rows[k], tile_rows);
    }
    a->unit_begin[kMaxW] = total;
    a->total_units = total;
}

void build_fused_units(const Plan& p, const ChunkRows& rows, int64_t tokens_per_unit,
                       int64_t block_tokens, int units_per_block, FusedArgs* a)
{
    const int W = p.W;
    a->W = W;
    a->d = int32_t(p.d);
    a->S = p.S;
    a->N = p.N;
    a->b = p.b;
    a->tokens_per_unit = int32_t(tokens_per_unit);
    a->block_tokens = int32_t(block_tokens);
    a->units_per_block = units_per_block;
    int64_t total = 0;  // blocks
    for (int k = 0; k < kMaxW; ++k) {
        const bool live = k < W;
        a->s[k] = live ? p.s[k] : 0;
        a->seq_off[k] = live ? p.seq_off[k] : 0;
        a->n[k] = live ? p.n[k] : 0;
        a->head_off[k] = live ? p.head_off[k] : 0;
        a->row_lo[k] = live ? rows.lo[k] : 0;
        a->rows[k] = live ? rows.cnt[k] : 0;
        a->unit_begin[k] = total;
        a->blocks[k] = live ? ceil_div(a->rows[k], block_tokens) : 0;
        total += p.b * a->blocks[k];
    }
    a->unit_begin[kMaxW] = total;
    a->total_units = total * units_per_block;
}

void build_fused_bwd_units(const Plan& p, const ChunkRows& rows, int64_t tokens_per_unit,
                           FusedBwdArgs* a)
{
    const int W = p.W;
    a->W = W;
    a->d = int32_t(p.d);
    a->S = p.S;
    a->N = p.N;
    a->b = p.b;
    a->tokens_per_unit = int32_t(tokens_per_unit);
    int64_t blocks = 0;
    for (int k = 0; k < kMaxW; ++k) {
        const bool live = k < W;
        a->s[k] = live ? p.s[k] : 0;
        a->seq_off[k] = live ? p.seq_off[k] : 0;
        a->n[k] = live ? p.n[k] : 0;
        a->head_off[k] = live ? p.head_off[k] : p.N;
        a->row_lo[k] = live ? rows.lo[k] : 0;
        a->rows[k] = live ? rows.cnt[k] : 0;
        a->block_begin[k] = blocks;
        a->blocks[k] = live ? ceil_div(a->rows[k], tokens_per_unit) : 0;
        blocks += p.b * a->blocks[k];
    }
    a->head_off[kMaxW] = p.N;
    a->block_begin[kMaxW] = blocks;
    a->total_units = int64_t(a->tensors) * blocks;
}

// theta^(-2j/d) expressed in turns (divided by 2 pi), split into a float pair whose sum carries
// about 48 significant bits, so that p * turn can be reduced modulo 1 exactly enough in fp32.
void rope_turns(int64_t d, double theta, float* turn_hi, float* turn_lo)
{
    const double two_pi = 6.283185307179586476925286766559;
    for (int64_t j = 0; j < d / 2; ++j) {
        const double t = std::pow(theta, -2.0 * double(j) / double(d)) / two_pi;
        const float hi = float(t);
        turn_hi[j] = hi;
        turn_lo[j] = float(t - double(hi));
    }
}

}  // namespace uly
