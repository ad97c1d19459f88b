/*
 * segment_memcpy.c -- a multi-threaded CPU relayout used only as a timed CPU baseline.
 *
 * TEST INFRASTRUCTURE, like the rest of this directory: only the benchmark's CPU-baseline leg and
 * the tests load it. It is not the oracle (the oracle is the element-by-element definition in
 * ulysses_oracle.c) and it is not the product: it is the relayout a CPU would run, written the
 * way the pages describe the operator (fast-ulysses 0.1.0, opening paragraph: the relayout is
 * expressed as copy strides, one contiguous run per token and destination rank), so that the
 * GPU's throughput can be set beside a reasonable multi-core host figure. The tests check that it
 * gives the oracle's bytes exactly.
 *
 * Mode 0: for every source shard q, batch index bb and row i, rank q's row (bb, i) holds W runs,
 * run r being n_r * d * e bytes at byte head_off(r) * d * e; run r is row seq_off(q) + i of rank
 * r's (b, S, n_r, d) tensor. Mode 1 copies the same runs the other way. Rows are cut into blocks
 * of up to 256, and the blocks are shared among OpenMP threads.
 */
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define SEG_MAX_W 8
#define SEG_BLOCK_ROWS 256

/* 0 on success, -1 on invalid arguments. threads <= 0: OpenMP's default. */
int seg_a2a_4d(int W, int64_t b, const int64_t* seq_splits, const int64_t* head_splits, int64_t d,
               int64_t e, int mode, const uint8_t* const* in, uint8_t* const* out, int threads)
{
    if (W < 1 || W > SEG_MAX_W || b < 1 || d < 1 || e < 1 || (mode != 0 && mode != 1)) return -1;
    int64_t seq_off[SEG_MAX_W + 1], head_off[SEG_MAX_W + 1], blocks_before[SEG_MAX_W + 1];
    seq_off[0] = head_off[0] = blocks_before[0] = 0;
    for (int k = 0; k < W; ++k) {
        if (seq_splits[k] < 0 || head_splits[k] < 0) return -1;
        seq_off[k + 1] = seq_off[k] + seq_splits[k];
        head_off[k + 1] = head_off[k] + head_splits[k];
        blocks_before[k + 1] =
            blocks_before[k] + b * ((seq_splits[k] + SEG_BLOCK_ROWS - 1) / SEG_BLOCK_ROWS);
    }
    const int64_t S = seq_off[W], N = head_off[W];
    if (S < 1 || N < 1) return -1;
    const int64_t row = N * d * e; /* one sequence-side row: all heads */
    const int64_t total = blocks_before[W];
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t blk = 0; blk < total; ++blk) {
        int q = 0;
        while (blocks_before[q + 1] <= blk) ++q;
        const int64_t per_batch = (seq_splits[q] + SEG_BLOCK_ROWS - 1) / SEG_BLOCK_ROWS;
        const int64_t local = blk - blocks_before[q];
        const int64_t bb = local / per_batch;
        const int64_t i0 = (local - bb * per_batch) * SEG_BLOCK_ROWS;
        const int64_t i1 = i0 + SEG_BLOCK_ROWS < seq_splits[q] ? i0 + SEG_BLOCK_ROWS : seq_splits[q];
        for (int64_t i = i0; i < i1; ++i) {
            const int64_t seq_at = (bb * seq_splits[q] + i) * row;
            for (int r = 0; r < W; ++r) {
                const int64_t run = head_splits[r] * d * e;
                if (run == 0) continue;
                const int64_t head_at = (bb * S + seq_off[q] + i) * run;
                const int64_t col = head_off[r] * d * e;
                if (mode == 0)
                    memcpy(out[r] + head_at, in[q] + seq_at + col, (size_t)run);
                else
                    memcpy(out[q] + seq_at + col, in[r] + head_at, (size_t)run);
            }
        }
    }
    return 0;
}

/* Threads an OpenMP parallel region of this library would use with threads <= 0. */
int seg_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
