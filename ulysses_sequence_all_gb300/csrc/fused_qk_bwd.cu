// fused_qk_bwd.cu -- backward of the fused QK call: the gradients of q, k and of the two RMSNorm
// weights from the gradients of the call's outputs, with the mode-1 gather fused in. The
// relayout is differentiable and its backward uses the forward's plan (fast-ulysses 0.2.1,
// README, "Quick start" and "Limits"; FastVideo, "Ulysses performance on GB200": backward uses
// the plan saved by its forward), and the backward of mode 0 is mode 1 on that plan.
//
// Forward, per head row x of d values at global sequence position p (fast-ulysses 0.1.0, "Fusion
// examples"): xh = x * r with r = 1 / sqrt(mean(x^2) + eps), y = R(p) (w * xh), where R(p)
// rotates each pair (2j, 2j+1) by p * theta^(-2j/d). For gy = dL/dy, in fp32:
//     u   = R(p)^T gy                          (the rotation by -p)
//     dw += u * xh                             (summed over every row of the tensor)
//     dx  = r * (u * w - xh * <u * w, xh> / d) = r * u * w - x * (r^3 <u * w, x> / d)
// dx is rounded once to bf16 and written on the sequence side, where x came from; gy is read
// on the head side, where mode 0 put y, so the rows arrive through the mode-1 gather.
//
// Structure: a persistent grid of several CTAs per SM, each with a ring of shared-memory stages;
// a loader warp (which also fills the rope table) and consumer warps. A unit is one tensor (q or
// k) of a block of tokens of one shard: the loader brings the forward input span (one bulk copy)
// and the output gradient (one bulk copy per token and rank: rank r's n_r heads, placed so that
// the gradient rows follow the input's (token, head) order) into a stage, decodes the unit once
// and leaves a small record of it beside the stage. The consumers compute dx row by row and store
// it from registers straight to the sequence side (16-byte stores; a token's rows are one
// contiguous span there, so the stores coalesce), then hand the stage back: a stage is held only
// while it loads and while it is computed, not while a store drains it. A group of 8 lanes holds
// a row (each lane 8 of its RoPE pairs; fused_row.cuh); three consumer warps share a unit's rows,
// and three CTAs with three stages each share an SM (at the Wan shape this measured faster than
// four CTAs of two stages, or four consumer warps of 16-lane rows). Each consumer lane keeps dw
// partial sums for its 16 columns; they are summed over the lanes of a warp when the tensor of
// its units changes (never for q, k alone with an even grid, where units alternate; once or twice
// for the interleaved call, whose units come in tensor phases) and at the end, and added to the
// warp's row of a small shared array; at the end the CTA's sums (over its warps, in a fixed
// order) fill its slot of a partial-sum array, which a second kernel adds up in a fixed order, so
// dw does not depend on timing. A v unit of the interleaved call (gradient rows only, mode 1)
// leaves by bulk stores from its stage.
//
// Row blocks (template flag GM; plans with equal head groups, runs of at most 2,048 bytes): a
// unit is a block of R whole rows of one tensor. Its forward input arrives with ONE 4-D tensor-map
// copy whose map walks (run, row, head group, batch), so it lands grouped by head group,
// [group][row][run], and each rank's gradient rows arrive as one span into the same order: 1 + W
// copies per R tokens instead of 1 + W per token. The consumers map a row (g, i, h) back to its
// sequence-side place (token i, head g n + h) for the dx store. One CTA per SM with 10 consumer
// warps and 2 stages of about 100 KiB.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/ulysses.h"
#include "fused_row.cuh"
#include "plan.h"
#include "ptx.cuh"

namespace uly {

static __device__ unsigned g_fused_bwd_status;

#ifndef ULY_BWD_CTAS_PER_SM
#define ULY_BWD_CTAS_PER_SM 3
#endif
#ifndef ULY_BWD_CONSUMER_WARPS
#define ULY_BWD_CONSUMER_WARPS 3
#endif
#ifndef ULY_BWD_STAGE_TARGET
#define ULY_BWD_STAGE_TARGET 20480
#endif
#ifndef ULY_BWD_MAX_STAGES
#define ULY_BWD_MAX_STAGES 3
#endif
#ifndef ULY_BWD_ILP
#define ULY_BWD_ILP 1
#endif
#ifndef ULY_BWD_WIDE  // 1: 8 RoPE pairs per lane for adjacent pairs too (fused_row.cuh)
#define ULY_BWD_WIDE 1
#endif
#ifndef ULY_BWD_WAIT_HINT_NS  // suspend-time hint of the barrier waits (0: plain polling)
#define ULY_BWD_WAIT_HINT_NS 10000
#endif
// Rotate-half pairs take 4 CTAs of 2 stages per SM (128 registers a thread, no spills): measured
// at the Wan-720p shape 0.984 / 0.977 of the copy peak (bf16 / fp16) against 0.953-0.967 with the
// adjacent pairs' 3 CTAs of 3 stages, which stay best for those (1.007 / 0.972 against 0.974 /
// 0.966).
#ifndef ULY_BWD_CTAS_PER_SM_HALF
#define ULY_BWD_CTAS_PER_SM_HALF 4
#endif
#ifndef ULY_BWD_MAX_STAGES_HALF
#define ULY_BWD_MAX_STAGES_HALF 2
#endif
constexpr int kBwdCtasPerSm = ULY_BWD_CTAS_PER_SM;
constexpr int kBwdMaxStages = ULY_BWD_MAX_STAGES;
constexpr int kBwdCtasPerSmHalf = ULY_BWD_CTAS_PER_SM_HALF;
constexpr int kBwdMaxStagesHalf = ULY_BWD_MAX_STAGES_HALF;
static_assert(kBwdMaxStagesHalf >= 2 && kBwdMaxStagesHalf <= kBwdMaxStages,
              "the barrier area holds kBwdMaxStages stages");
constexpr int kBwdNW = ULY_BWD_CONSUMER_WARPS;
constexpr int kBwdIlp = ULY_BWD_ILP;  // head rows in flight per lane group
#ifndef ULY_BWD_ILP_WIDE  // the same for the 8-pair row layout (rotate half), twice the values
#define ULY_BWD_ILP_WIDE 1
#endif
constexpr int kBwdIlpWide = ULY_BWD_ILP_WIDE;
constexpr bool kBwdWide = ULY_BWD_WIDE != 0;
constexpr int kBwdHeader = 256;  // two barriers per stage, then one unit record per stage
constexpr int kBwdRecordsAt = 128;
static_assert(2 * 8 * kBwdMaxStages <= kBwdRecordsAt, "stage barriers must fit the header");
static_assert(kBwdRecordsAt + 16 * kBwdMaxStages <= kBwdHeader, "unit records must fit");
// Row blocks (group-major units, plans with equal head groups): one CTA per SM with 10 consumer
// warps, blocks of max(3, ULY_BWD_GM_BYTES / row) rows, 2 stages. Measured at the Wan-720p shape
// 1.014-1.029 of the copy peak in all four element and pair layouts (token units 0.972-1.004);
// 8, 9, 12 or 14 consumer warps, 3-row blocks in 3 stages or 2-row blocks measured 0.82-0.98.
#ifndef ULY_BWD_GM_WARPS
#define ULY_BWD_GM_WARPS 10
#endif
#ifndef ULY_BWD_GM_BYTES
#define ULY_BWD_GM_BYTES 51200
#endif
#ifndef ULY_BWD_GM_MIN_ROWS
#define ULY_BWD_GM_MIN_ROWS 3
#endif
#ifndef ULY_BWD_GM_STAGES
#define ULY_BWD_GM_STAGES 2
#endif
constexpr int kBwdNWGm = ULY_BWD_GM_WARPS;
static_assert(ULY_BWD_GM_STAGES >= 2 && ULY_BWD_GM_STAGES <= kBwdMaxStages, "stage barriers");
constexpr int kBwdLoaderWarp = 0, kBwdFirstConsumer = 1;
__host__ __device__ constexpr int bwd_warps(bool gm) { return gm ? kBwdNWGm : kBwdNW; }
__host__ __device__ constexpr int bwd_threads(bool gm)
{
    return 32 * (kBwdFirstConsumer + bwd_warps(gm));
}
constexpr int kBwdConsumerBarrier = 1;  // named barrier of the consumer warps (0: __syncthreads)

struct BwdUnit {
    int t;  // 0: q, 1: k, 2 ..: the packed call's other planes (gradient gathered by mode 1)
    int q;
    int64_t bb, i0;
    int ntok;
};

// What the consumers and the storer need of a unit, written by the loader next to the stage
// before it arrives on "full" (the loader decodes each unit once).
struct BwdRecord {
    int64_t seq_row0;  // first row (token) of the unit in rank q's (b, s_q) sequence side
    int32_t t_q;       // tensor (bits 0-2) and shard q (bits 3..)
    int32_t ntok;
};

__device__ __forceinline__ bool bwd_wait(uint64_t* bar, uint32_t parity)
{
#if ULY_BWD_WAIT_HINT_NS > 0
    return mbar_wait_bounded_hint<ULY_BWD_WAIT_HINT_NS>(bar, parity);
#else
    return mbar_wait_bounded(bar, parity);
#endif
}

__device__ __forceinline__ BwdUnit bwd_decode(const FusedBwdArgs& a, int64_t u)
{
    BwdUnit x;
    int64_t blk_id;
    if (a.tensors == 2) {  // q and k units alternate
        blk_id = u >> 1;
        x.t = int(u & 1);
    } else {  // packed: every q unit, then every k unit, then each other plane's units (for QKV
              // the alternating order measured 2% slower, and 1% faster for q, k alone)
        const int64_t blocks_all = a.block_begin[kMaxW];
        x.t = int(div_fast(u, blocks_all));
        blk_id = u - int64_t(x.t) * blocks_all;
    }
    int lo = 0, hi = a.W - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.block_begin[mid] <= blk_id)
            lo = mid;
        else
            hi = mid - 1;
    }
    x.q = lo;
    const int64_t T = a.tokens_per_unit;
    const int64_t blocks = a.blocks[lo];  // token blocks per batch index of shard q
    const int64_t local = blk_id - a.block_begin[lo];
    x.bb = div_fast(local, blocks);
    const int64_t blk = local - x.bb * blocks;
    x.i0 = a.row_lo[lo] + blk * T;
    x.ntok = int(min(T, a.rows[lo] - blk * T));
    return x;
}

// Shared-memory layout (byte offsets), shared by the kernel and its launcher.
struct BwdSmem {
    int turns;   // float2 (hi, lo) per pair j < d/2
    int tables;  // per stage: (cos, sin) per (token, pair)
    int weights; // 2 x d fp32 RMSNorm weights
    int red;     // per consumer warp: 2 x d fp32 dw sums
    int stages;  // per stage: forward input span, then output-gradient runs
    int table_bytes;
    int total;
};

__host__ __device__ inline BwdSmem bwd_smem_layout(int d, int tokens, int stages,
                                                   uint32_t stage_bytes, int nw)
{
    auto up = [](int x) { return (x + 127) & ~127; };
    BwdSmem m;
    m.turns = kBwdHeader;
    m.tables = up(m.turns + (d / 2) * 8);
    m.table_bytes = up(tokens * (d / 2) * 8);
    m.weights = up(m.tables + stages * m.table_bytes);
    m.red = m.weights + 2 * d * 4;
    m.stages = up(m.red + nw * 2 * d * 4);
    m.total = m.stages + stages * int(stage_bytes);
    return m;
}

// Rows of dw sums per consumer warp in shared memory (each 2 x d floats, q then k): one per row
// group of the warp where rows are packed back to back in the warp (a run-time layout whose
// row_lane_stride is not a power of two; each lane then adds its sums to its group's row, no
// shuffle), else one (the warp's groups summed with a butterfly first).
__host__ __device__ inline int bwd_dw_rows_per_warp(int d)
{
    if ((d & (d - 1)) == 0) return 1;
    const int g = d / (d % 16 == 0 ? 16 : 8);
    const int gp = row_lane_stride(g);
    return (gp & (gp - 1)) == 0 ? 1 : 32 / g;
}

// D: head dimension, a power of two, or below 8 for a.d with one of the run-time row layouts
// (rt_layout_for: any multiple of 8 up to 256); F16: fp16 elements (else bf16); HALF_PAIRS:
// rotate-half RoPE pairs (else adjacent pairs). The row layouts (G lanes per row, H packed slots
// per lane) are in fused_row.cuh.
template <int D, bool F16, bool HALF_PAIRS, bool GM>
__global__ void __launch_bounds__(bwd_threads(GM),
                                  GM ? 1 : HALF_PAIRS ? kBwdCtasPerSmHalf : kBwdCtasPerSm)
    fused_qk_bwd_kernel(const __grid_constant__ FusedBwdArgs a)
{
    constexpr int kNW = bwd_warps(GM);  // consumer warps
    using IO = RowIO<F16, HALF_PAIRS, D, kBwdWide>;
    using Words = typename IO::Words;
    const int dd = rt_layout(D) ? a.d : D;  // head dimension
    const RowDims dims = IO::dims(dd);
    const int G = dims.g;        // lanes per head row
    constexpr int H = IO::H;
    const int HALF = dd / 2;
    // lanes from a row's first to the next row's: G, or G rounded up to a power of two
    const int GP = !rt_layout(D) ? G : rt_pow2(D) ? row_lane_stride(G) : G;
    const int GPW = 32 / GP;  // head rows per warp per slot
    // rows in flight per lane group: a lane of an 8-pair layout holds twice the values
    constexpr int ILP = IO::P == 8 ? kBwdIlpWide : kBwdIlp;
    const int PER_STEP = GPW * ILP;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int K = a.stages;
    const int N = int(a.N);
    const int RG = rt_layout(D) ? bwd_dw_rows_per_warp(dd) : 1;  // dw rows per consumer warp
    const BwdSmem L = bwd_smem_layout(dd, a.tokens_per_unit, K, a.stage_bytes, kNW * RG);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);  // data landed + table written
    uint64_t* empty = full + kBwdMaxStages;              // consumers done with the stage
    float2* turns = reinterpret_cast<float2*>(smem + L.turns);
    float* red = reinterpret_cast<float*>(smem + L.red);
    float* wsm = reinterpret_cast<float*>(smem + L.weights);
    BwdRecord* records = reinterpret_cast<BwdRecord*>(smem + kBwdRecordsAt);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t first = blockIdx.x, step = gridDim.x;
    const int64_t n = first < a.total_units ? (a.total_units - 1 - first) / step + 1 : 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < K; ++s) {
            mbar_init(&full[s], 1 + 32);  // the loader's expect_tx, then its lanes' table writes
            mbar_init(&empty[s], kNW);
        }
        fence_barrier_init();
    }
    for (int j = threadIdx.x; j < HALF; j += blockDim.x) turns[j] = make_float2(a.turn_hi[j], a.turn_lo[j]);
    for (int j = threadIdx.x; j < kNW * RG * 2 * dd; j += blockDim.x) red[j] = 0.0f;
    for (int j = threadIdx.x; j < 2 * dd; j += blockDim.x) wsm[j] = a.rms_w[j];
    __syncthreads();
    const int row_bytes = N * dd * 2;               // one token, all heads, one tensor
    const uint32_t grad_at = a.stage_bytes / 2;     // the gradient runs' offset in a stage
    const bool packed_rows = a.tok_stride == row_bytes;  // a block's rows are one span

    if (warp == kBwdLoaderWarp) {
        // Per unit: lane 0 the input span (one copy per token when the tokens are interleaved
        // with other planes); then one copy per (token, rank) of the gradient, so that the
        // gradient rows land in the input's (token, head) order, grad_at bytes further. A v unit
        // (interleaved QKV) has no input: its gradient rows land at the start of the stage and
        // leave unchanged (mode 1).
        int64_t j = 0;
        StageRing ring;
        for (; j < n; ++j, ring.next(K)) {
            const int s = ring.s;
            int ok = 1;
            if (lane == 0 && j >= K) ok = bwd_wait(&empty[s], ring.phase ^ 1u);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) atomicOr(&g_fused_bwd_status, kStatusWaitTimeout);
                break;
            }
            const BwdUnit t = bwd_decode(a, first + j * step);
            const bool is_v = t.t >= 2;
            const uint32_t span = uint32_t(t.ntok) * uint32_t(row_bytes);
            uint8_t* dst = smem + L.stages + size_t(s) * a.stage_bytes;
            const int64_t tok0 = t.bb * a.s[t.q] + t.i0;
            const int64_t row0 = t.bb * a.S + a.seq_off[t.q] + t.i0;  // first head-side row
            if (GM && !is_v) {
                // the input block, grouped by head group (R whole rows arrive: rows past the
                // chunk are filled), then each rank's gradient rows as one span, in the same order
                if (lane == 0) {
                    const uint32_t box = uint32_t(a.tokens_per_unit) * uint32_t(row_bytes);
                    mbar_arrive_expect_tx(&full[s], box + uint32_t(t.ntok) * a.run * uint32_t(a.W));
                    tensor_g2s_4d(dst, &a.xmap[t.t][t.q], 0, int(t.i0 - a.row_lo[t.q]), 0,
                                  int(t.bb), &full[s]);
                    BwdRecord& rec = records[s];  // published by this lane's arrive below
                    rec.seq_row0 = tok0;
                    rec.t_q = t.t | (t.q << 3);
                    rec.ntok = t.ntok;
                }
                __syncwarp();  // the unit's bytes are registered before any copy can complete
                if (lane < a.W)
                    bulk_g2s(dst + grad_at + size_t(lane) * a.tokens_per_unit * a.run,
                             a.g_in[t.t][lane] + row0 * a.run, uint32_t(t.ntok) * a.run, &full[s]);
            }
            if (lane == 0 && !GM) {
                mbar_arrive_expect_tx(&full[s], is_v ? span : 2 * span);
                if (!is_v && packed_rows)
                    bulk_g2s(dst, a.x_in[t.t][t.q] + tok0 * row_bytes, span, &full[s]);
                BwdRecord& rec = records[s];  // published by this lane's arrive below
                rec.seq_row0 = tok0;
                rec.t_q = t.t | (t.q << 3);
                rec.ntok = t.ntok;
            }
            __syncwarp();
            if (!GM && !is_v && !packed_rows) {
                for (int tok = lane; tok < t.ntok; tok += 32)
                    bulk_g2s(dst + tok * row_bytes, a.x_in[t.t][t.q] + (tok0 + tok) * a.tok_stride,
                             uint32_t(row_bytes), &full[s]);
            }
            if (GM && is_v) {  // each rank's rows as one span, grouped by head group as well
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full[s], uint32_t(t.ntok) * a.run * uint32_t(a.W));
                    BwdRecord& rec = records[s];  // published by this lane's arrive below
                    rec.seq_row0 = tok0;
                    rec.t_q = t.t | (t.q << 3);
                    rec.ntok = t.ntok;
                }
                __syncwarp();  // the unit's bytes are registered before any copy can complete
                if (lane < a.W)
                    bulk_g2s(dst + size_t(lane) * a.tokens_per_unit * a.run,
                             a.g_in[t.t][lane] + row0 * a.run, uint32_t(t.ntok) * a.run, &full[s]);
            }
            uint8_t* gdst = is_v ? dst : dst + grad_at;
            const int copies = GM ? 0 : t.ntok * a.W;  // token order: one per (token, rank)
            for (int c = lane; c < copies; c += 32) {
                const int tok = c / a.W, r = c - tok * a.W;
                const int64_t run = a.n[r] * (dd * 2);  // bytes per token on rank r
                if (run == 0) continue;
                bulk_g2s(gdst + tok * row_bytes + int(a.head_off[r]) * (dd * 2),
                         a.g_in[t.t][r] + (row0 + tok) * run, uint32_t(run), &full[s]);
            }
            // While the copies fly, the lanes fill the stage's cos/sin table for the unit's
            // positions (free: the stage's previous unit has been consumed) and arrive on "full",
            // so a consumer that sees the phase complete sees both.
            // Per token, lane i of a row group reads P / 2 16-byte entries (c_j, c_j+1, s_j,
            // s_j+1), j = P i + 2h; for each h the entries of all lanes are adjacent.
            float* table = reinterpret_cast<float*>(smem + L.tables + s * L.table_bytes);
            const float p0 = float(a.seq_off[t.q] + t.i0);
            for (int e = lane; e < (is_v ? 0 : t.ntok * HALF); e += 32) {
                const int tok = e / HALF, jj = e % HALF;
                const float2 tj = turns[jj];
                const float2 cs = rope_cos_sin(p0 + float(tok), tj.x, tj.y);
                const int at = IO::table_at(tok, jj, dims);
                table[at] = cs.x;
                table[at + 2] = cs.y;
            }
            mbar_arrive(&full[s]);
        }
        // do not leave while copies into this CTA's shared memory may be in flight
        if (lane == 0) {
            for (int64_t jj = (j > K ? j - K : 0); jj < j; ++jj) {
                if (!mbar_wait_bounded(&full[jj % K], uint32_t((jj / K) & 1))) {
                    atomicOr(&g_fused_bwd_status, kStatusDrainTimeout);
                    break;
                }
            }
        }
        return;
    }

    // consumers: all warps work on the unit's tensor, each on a contiguous share of its rows. A
    // group of G lanes holds one head row (a lane's RoPE pairs as packed fp32 values: the first
    // and the second elements of its pairs), ILP rows in flight per group.
    const int cw = warp - kBwdFirstConsumer;
    const int group = lane / GP;       // which head row of the warp slot
    const int sub = lane - group * GP;  // which pairs of the row this lane holds
    const bool active = sub < G && group < GPW;  // lanes holding no row's pairs (run-time d)
    const float inv_d = 1.0f / float(dd);
    // dw partial sums of this lane's columns for tensor acc_t, flushed when the tensor changes
    // (with an even grid a CTA of the q, k call only ever sees one tensor) and at the end
    float2 aE[H], aO[H];
#pragma unroll
    for (int h = 0; h < H; ++h) aE[h] = aO[h] = make_float2(0.f, 0.f);
    int acc_t = -1;
    bool stored_v = false;  // this lane issued bulk stores (v units) that must finish before exit
    // this warp's share of the rows of a full token block (steps m_lo .. m_hi - 1 of PER_STEP
    // rows), and the (token, head) of its first row
    const int full_steps = (a.tokens_per_unit * N + PER_STEP - 1) / PER_STEP;
    const int full_m_lo = cw * full_steps / kNW, full_m_hi = (cw + 1) * full_steps / kNW;
    const int full_base_tok = full_m_lo * PER_STEP / N;
    const int full_base_head = full_m_lo * PER_STEP - full_base_tok * N;
    // group-major units: row (group g, row i, head h) at ((g R + i) n + h) in both halves of the
    // stage, the same share of steps for every unit (short units skip rows past their end)
    const int gm_n = GM ? a.n_eq : 1, gm_R = a.tokens_per_unit;
    const int gm_run = GM ? int(a.run) : 0;
    const int gm_pt0 = full_m_lo * PER_STEP / gm_n;  // pseudo-token g R + i of the first row
    const int gm_h0 = full_m_lo * PER_STEP - gm_pt0 * gm_n;
    const int gm_g0 = gm_pt0 / gm_R, gm_i0 = gm_pt0 - (gm_pt0 / gm_R) * gm_R;
    // sums over the lane groups of the warp, added to the warp's shared row, then cleared
    auto flush_dw = [&]() {
        if constexpr (rt_pow2(D)) {  // rows on power-of-two strides: sum the groups, then group 0
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                if (off < GP) continue;  // across the warp's row groups, not within a row
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    aE[h].x += __shfl_xor_sync(0xffffffffu, aE[h].x, off);
                    aE[h].y += __shfl_xor_sync(0xffffffffu, aE[h].y, off);
                    aO[h].x += __shfl_xor_sync(0xffffffffu, aO[h].x, off);
                    aO[h].y += __shfl_xor_sync(0xffffffffu, aO[h].y, off);
                }
            }
        }
        // rows packed back to back: every group adds to its own row
        const int rg = rt_pow2(D) ? 0 : group;
        if ((rt_pow2(D) ? group == 0 : true) && active && acc_t >= 0) {
            float* row = red + ((cw * RG + rg) * 2 + acc_t) * dd;
#pragma unroll
            for (int h = 0; h < H; ++h) {
                row[IO::col(sub, h, false, 0, dims)] += aE[h].x;
                row[IO::col(sub, h, true, 0, dims)] += aO[h].x;
                row[IO::col(sub, h, false, 1, dims)] += aE[h].y;
                row[IO::col(sub, h, true, 1, dims)] += aO[h].y;
            }
        }
#pragma unroll
        for (int h = 0; h < H; ++h) {
            aE[h] = make_float2(0.f, 0.f);
            aO[h] = make_float2(0.f, 0.f);
        }
    };
    StageRing ring;
    for (int64_t k = 0; k < n; ++k, ring.next(K)) {
        const int s = ring.s;
        if (!__all_sync(0xffffffffu, bwd_wait(&full[s], ring.phase))) {
            if (lane == 0) atomicOr(&g_fused_bwd_status, kStatusWaitTimeout);
            break;
        }
        const BwdRecord rec = records[s];
        const int tt = rec.t_q & 7, ntok = rec.ntok;
        uint8_t* xs = smem + L.stages + size_t(s) * a.stage_bytes;
        if (tt >= 2) {  // another plane's unit: its rows leave as they came (mode 1), stored
                        // by the first consumer warp
            if (cw == 0 && lane == 0) {
                uint8_t* out = a.dx_out[tt][rec.t_q >> 3] + rec.seq_row0 * a.tok_stride;
                if (GM) {  // grouped by head group: one tensor-map store back to token order
                    const int q = rec.t_q >> 3;
                    const int64_t bb = rec.seq_row0 / a.s[q];
                    const int64_t i0 = rec.seq_row0 - bb * a.s[q] - a.row_lo[q];
                    tensor_s2g_4d(&a.dmap[tt - 2][q], 0, int(i0), 0, int(bb), xs);
                } else if (packed_rows) {
                    bulk_s2g(out, xs, uint32_t(ntok) * uint32_t(row_bytes));
                } else {
                    for (int tok = 0; tok < ntok; ++tok)
                        bulk_s2g(out + int64_t(tok) * a.tok_stride, xs + tok * row_bytes,
                                 uint32_t(row_bytes));
                }
                bulk_commit();
                bulk_wait_read<0>();  // the stage may be refilled once the store has read it
                stored_v = true;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            continue;
        }
        float2 wE[H], wO[H];  // this lane's weights of the unit's tensor (first / second elements)
#pragma unroll
        for (int h = 0; h < H; ++h) wE[h] = wO[h] = make_float2(0.f, 0.f);
        if (active) IO::weights(wsm + tt * dd, sub, wE, wO, dims);
        const uint8_t* gs = xs + grad_at;
        uint8_t* out_base = a.dx_out[tt][rec.t_q >> 3] + rec.seq_row0 * a.tok_stride;
        const float4* table = reinterpret_cast<const float4*>(smem + L.tables + s * L.table_bytes);
        if (tt != acc_t) {  // the sums so far belong to the other tensor
            flush_dw();
            acc_t = tt;
        }
        const int rows = ntok * N;
        int m_lo = full_m_lo, m_hi = full_m_hi;
        int base_tok = full_base_tok, base_head = full_base_head;
        if (!GM && ntok != a.tokens_per_unit) {  // a short block: this warp's share of its rows
            const int steps = (rows + PER_STEP - 1) / PER_STEP;
            m_lo = cw * steps / kNW;
            m_hi = (cw + 1) * steps / kNW;
            base_tok = m_lo * PER_STEP / N;
            base_head = m_lo * PER_STEP - base_tok * N;
        }
        int base = m_lo * PER_STEP;  // first row of the current step and its (token, head)
        int bg = gm_g0, bi = gm_i0, bh = gm_h0;  // group-major: (group, row, head) of the step
        for (int m = m_lo; m < m_hi; ++m) {
            // The sums (mean square, <u * w, x>) need the whole row: u = R^T gy (fp32) and the
            // raw words of x are kept across the reduction, then dx and the dw terms are formed.
            int tk_[ILP], hh_[ILP];
            bool ok[ILP];
            Words xr[ILP];
            float2 uE[ILP][H], uO[ILP][H];
            float ss[ILP], dp[ILP];
#pragma unroll
            for (int u = 0; u < ILP; ++u) {
                const int o = u * GPW + group;
                int off;  // the row's offset in both halves of the stage
                if constexpr (GM) {
                    int hh = bh + o, ii = bi, gg = bg;
                    while (hh >= gm_n) {
                        hh -= gm_n;
                        if (++ii == gm_R) {
                            ii = 0;
                            ++gg;
                        }
                    }
                    ok[u] = gg < a.W && ii < ntok;
                    tk_[u] = ii;
                    hh_[u] = gg * gm_n + hh;  // head on the sequence side
                    off = (gg * gm_R + ii) * gm_run + hh * (dd * 2);
                } else {
                    ok[u] = base + o < rows;
                    int hh = base_head + o, tk = base_tok;
                    while (hh >= N) {
                        hh -= N;
                        ++tk;
                    }
                    tk_[u] = tk;
                    hh_[u] = hh;
                    off = (base + o) * (dd * 2);  // row (tk, hh) of the unit in the stage
                }
                Words g = {};
                xr[u] = Words{};
                if (ok[u] && active) {
                    xr[u] = IO::load(xs + off, sub, dims);
                    g = IO::load(gs + off, sub, dims);
                }
                float2 acc_ss = make_float2(0.f, 0.f), acc_dp = make_float2(0.f, 0.f);
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    float2 xE, xO, gE, gO;  // first / second elements of the lane's pairs
                    IO::unpack(xr[u], h, xE, xO);
                    IO::unpack(g, h, gE, gO);
                    // (c_j, c_j+1, s_j, s_j+1) for j = P sub + 2 h
                    const float4 cs = active ? table[IO::table_entry(tk_[u], h, sub, dims)]
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                    const float2 c2 = make_float2(cs.x, cs.y), s2 = make_float2(cs.z, cs.w);
                    const float2 ns2 = make_float2(-cs.z, -cs.w);
                    // u = R^T gy: (c g_e + s g_o, c g_o - s g_e)
                    uE[u][h] = __ffma2_rn(gO, s2, __fmul2_rn(gE, c2));
                    uO[u][h] = __ffma2_rn(gE, ns2, __fmul2_rn(gO, c2));
                    acc_ss = __ffma2_rn(xE, xE, acc_ss);
                    acc_ss = __ffma2_rn(xO, xO, acc_ss);
                    acc_dp = __ffma2_rn(__fmul2_rn(uE[u][h], wE[h]), xE, acc_dp);
                    acc_dp = __ffma2_rn(__fmul2_rn(uO[u][h], wO[h]), xO, acc_dp);
                }
                ss[u] = acc_ss.x + acc_ss.y;
                dp[u] = acc_dp.x + acc_dp.y;
            }
            row_sums<D, 2>(ss, dp, G, GP, sub, group);
#pragma unroll
            for (int u = 0; u < ILP; ++u) {
                if (!ok[u] || !active) continue;
                const float rr = rsqrtf(ss[u] * inv_d + a.eps);
                const float kk = rr * rr * rr * dp[u] * inv_d;
                const float2 r2 = make_float2(rr, rr), nk2 = make_float2(-kk, -kk);
                float2 dxE[H], dxO[H];
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    float2 xE, xO;
                    IO::unpack(xr[u], h, xE, xO);
                    dxE[h] = __ffma2_rn(__fmul2_rn(uE[u][h], wE[h]), r2, __fmul2_rn(xE, nk2));
                    dxO[h] = __ffma2_rn(__fmul2_rn(uO[u][h], wO[h]), r2, __fmul2_rn(xO, nk2));
                    aE[h] = __ffma2_rn(uE[u][h], __fmul2_rn(xE, r2), aE[h]);
                    aO[h] = __ffma2_rn(uO[u][h], __fmul2_rn(xO, r2), aO[h]);
                }
                // straight to the sequence side: row (token, head) of this unit's dx
                IO::store_global(out_base + int64_t(tk_[u]) * a.tok_stride + hh_[u] * (dd * 2), sub,
                                 IO::pack(dxE, dxO), dims);
            }
            if constexpr (GM) {
                bh += PER_STEP;
                while (bh >= gm_n) {
                    bh -= gm_n;
                    if (++bi == gm_R) {
                        bi = 0;
                        ++bg;
                    }
                }
            } else {
                base += PER_STEP;
                base_head += PER_STEP;
                while (base_head >= N) {
                    base_head -= N;
                    ++base_tok;
                }
            }
        }
        // this warp has read all it needs of the stage: hand it back
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    flush_dw();
    if (stored_v) bulk_wait<0>();
    // the CTA's dw sums, over its consumer warps in a fixed order, into its slot
    asm volatile("bar.sync %0, %1;" ::"r"(kBwdConsumerBarrier), "r"(kNW * 32) : "memory");
    const int ct = threadIdx.x - kBwdFirstConsumer * 32;
    float* slot_out = a.dw_part + size_t(blockIdx.x) * (2 * dd);
    for (int j = ct; j < 2 * dd; j += kNW * 32) {
        float sum = 0.0f;
        for (int w = 0; w < kNW * RG; ++w) sum += red[w * 2 * dd + j];
        slot_out[j] = sum;
    }
}

// dw[j] = (dw[j] if accumulate) + the sum over slots c < slots of part[c][j], j < n, in a fixed
// order: warp w of a block adds slots w, w + 16, ... for 32 columns, then warp 0 adds the 16.
__global__ void __launch_bounds__(512) fused_bwd_reduce_kernel(const float* __restrict__ part,
                                                               int slots, int n,
                                                               float* __restrict__ dw,
                                                               int accumulate)
{
    __shared__ float acc[16][33];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int j = blockIdx.x * 32 + lane;
    float s = 0.0f;
    if (j < n) {
        for (int c = w; c < slots; c += 16) s += part[size_t(c) * n + j];
    }
    acc[w][lane] = s;
    __syncthreads();
    if (w == 0 && j < n) {
        float total = 0.0f;
        for (int k = 0; k < 16; ++k) total += acc[k][lane];
        dw[j] = accumulate ? dw[j] + total : total;
    }
}

// Stage geometry for a plan: tokens per unit, stage count and CTAs per SM (0 stages: one token's
// input and gradient rows do not fit even one CTA per SM). Narrower units, fewer stages, then
// fewer CTAs per SM are tried in that order.
// Whether the backward takes row blocks under the automatic choice (the plan must fit them:
// equal head groups, runs of at most 2,048 bytes). Measured across eight plans with equal head
// groups (CUDA events, back to back): with rows of 7-16 KiB they ran at 1.006-1.034 of the copy
// peak against the token units' 0.78-1.00; with 4 KiB rows (N d e = 4,096) at 0.81-0.88 against
// 0.76-0.94, mostly below.
bool fused_bwd_group_major_preferred(const Plan& p) { return p.N * p.d * p.e >= 6144; }

void fused_bwd_geometry(const Plan& p, bool group_major, int64_t* tokens_per_unit, int* stages,
                        uint32_t* stage_bytes, int* ctas_per_sm)
{
    *stages = 0;
    *tokens_per_unit = 1;
    *stage_bytes = 0;
    *ctas_per_sm = 1;
    const int64_t row = p.N * p.d * 2;  // one token of one tensor
    if (group_major) {  // one CTA per SM; the largest block (at least the target) that fits
        int64_t R = ULY_BWD_GM_BYTES / row;
        if (R < ULY_BWD_GM_MIN_ROWS) R = ULY_BWD_GM_MIN_ROWS;
        if (R > 256) R = 256;
        for (; R >= 1; --R) {
            const int64_t half = (R * row + 127) / 128 * 128;  // input box, then gradient rows
            if (2 * half >= (1 << 20)) continue;
            const BwdSmem m = bwd_smem_layout(int(p.d), int(R), ULY_BWD_GM_STAGES,
                                              uint32_t(2 * half),
                                              kBwdNWGm * bwd_dw_rows_per_warp(int(p.d)));
            if (m.total <= kSmemPerCtaMax) {
                *tokens_per_unit = R;
                *stages = ULY_BWD_GM_STAGES;
                *stage_bytes = uint32_t(2 * half);
                *ctas_per_sm = 1;
                return;
            }
        }
        return;
    }
    const int64_t tok_bytes = 2 * row;  // one token's input and gradient rows
    int64_t T0 = ULY_BWD_STAGE_TARGET / tok_bytes;
    if (T0 < 1) T0 = 1;
    const int ctas_max = p.rope_half ? kBwdCtasPerSmHalf : kBwdCtasPerSm;
    const int stages_max = p.rope_half ? kBwdMaxStagesHalf : kBwdMaxStages;
    for (int ctas = ctas_max; ctas >= 1; --ctas) {
        const int budget = kSmemPerSm / ctas - kSmemReservedPerCta;
        for (int64_t T = T0; T >= 1; T = T > 1 ? T / 2 : 0) {
            const int64_t sb = T * tok_bytes;
            if (sb >= (1 << 20)) continue;  // an mbarrier counts fewer than 2^20 bytes
            for (int K = stages_max; K >= 2; --K) {
                const BwdSmem m = bwd_smem_layout(int(p.d), int(T), K, uint32_t(sb),
                                                  kBwdNW * bwd_dw_rows_per_warp(int(p.d)));
                if (m.total <= budget && m.total <= kSmemPerCtaMax) {
                    *tokens_per_unit = T;
                    *stages = K;
                    *stage_bytes = uint32_t(sb);
                    *ctas_per_sm = ctas;
                    return;
                }
            }
        }
    }
}

template <int D, bool F16, bool HALF, bool GM>
static cudaError_t bwd_launch_d(const FusedBwdArgs& a, cudaStream_t stream, int device, int grid)
{
    static std::atomic<unsigned long long> raised{0};  // devices with this variant's limit raised
    const unsigned long long bit = device >= 0 && device < 64 ? 1ull << device : 0;
    if (bit && !(raised.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(fused_qk_bwd_kernel<D, F16, HALF, GM>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemPerCtaMax);
        if (e != cudaSuccess) return e;
        raised.fetch_or(bit);
    }
    const BwdSmem m =
        bwd_smem_layout(a.d, a.tokens_per_unit, a.stages, a.stage_bytes,
                        bwd_warps(GM) * bwd_dw_rows_per_warp(a.d));
    fused_qk_bwd_kernel<D, F16, HALF, GM><<<grid, bwd_threads(GM), m.total, stream>>>(a);
    return cudaGetLastError();
}

template <int D, bool F16, bool HALF>
static cudaError_t bwd_launch_gm(const FusedBwdArgs& a, cudaStream_t stream, int device, int grid)
{
    return a.group_major ? bwd_launch_d<D, F16, HALF, true>(a, stream, device, grid)
                         : bwd_launch_d<D, F16, HALF, false>(a, stream, device, grid);
}

template <int D>
static cudaError_t bwd_launch_variant(const FusedBwdArgs& a, cudaStream_t stream, int device,
                                      int grid)
{
    if (a.elem_f16)
        return a.rope_half ? bwd_launch_gm<D, true, true>(a, stream, device, grid)
                           : bwd_launch_gm<D, true, false>(a, stream, device, grid);
    return a.rope_half ? bwd_launch_gm<D, false, true>(a, stream, device, grid)
                       : bwd_launch_gm<D, false, false>(a, stream, device, grid);
}

// CTAs of the main kernel for a launch of `a` (the number of partial-sum slots it fills); at
// most max_grid when that is positive.
int64_t fused_bwd_grid(const FusedBwdArgs& a, int sm_count, int64_t max_grid)
{
    int64_t grid = int64_t(sm_count) * (a.ctas_per_sm > 0 ? a.ctas_per_sm : 1);
    if (max_grid > 0 && grid > max_grid) grid = max_grid;
    return grid < a.total_units ? grid : a.total_units;
}

// One launch of the backward over `a` (its dw_part holds at least fused_bwd_grid slots), then
// the reduction of its slots into dw (added to dw when `accumulate`, else written).
cudaError_t fused_bwd_launch(const FusedBwdArgs& a, float* dw, bool accumulate, cudaStream_t stream,
                             int device, int sm_count, int64_t max_grid)
{
    const int64_t grid = fused_bwd_grid(a, sm_count, max_grid);
    if (grid > 0) {
        cudaError_t e;
        switch (a.d) {
            case 8: e = bwd_launch_variant<8>(a, stream, device, int(grid)); break;
            case 16: e = bwd_launch_variant<16>(a, stream, device, int(grid)); break;
            case 32: e = bwd_launch_variant<32>(a, stream, device, int(grid)); break;
            case 64: e = bwd_launch_variant<64>(a, stream, device, int(grid)); break;
            case 128: e = bwd_launch_variant<128>(a, stream, device, int(grid)); break;
            case 256: e = bwd_launch_variant<256>(a, stream, device, int(grid)); break;
            default:  // any other multiple of 8 up to 256: a run-time row layout
                if (a.d % 8 != 0 || a.d < 8 || a.d > kMaxFusedD) return cudaErrorInvalidValue;
                switch (rt_layout_for(a.d)) {
                    case 0: e = bwd_launch_variant<0>(a, stream, device, int(grid)); break;
                    case kRtWide: e = bwd_launch_variant<kRtWide>(a, stream, device, int(grid)); break;
                    case kRtPow2: e = bwd_launch_variant<kRtPow2>(a, stream, device, int(grid)); break;
                    default:
                        e = bwd_launch_variant<kRtPow2 | kRtWide>(a, stream, device, int(grid));
                        break;
                }
                break;
        }
        if (e != cudaSuccess) return e;
    } else if (accumulate) {
        return cudaSuccess;  // nothing to add
    }
    const int n = 2 * a.d;
    fused_bwd_reduce_kernel<<<(n + 31) / 32, 512, 0, stream>>>(a.dw_part, int(grid), n, dw,
                                                              accumulate ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t fused_bwd_status(unsigned* status, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(status, g_fused_bwd_status, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_fused_bwd_status, &zero, sizeof(unsigned));
}

}  // namespace uly
