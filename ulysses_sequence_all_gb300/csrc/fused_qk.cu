// fused_qk.cu -- mode-0 relayout of q and k with QK RMSNorm + RoPE applied in the scatter
// (fast-ulysses 0.1.0, "Fusion examples": QK RMSNorm + RoPE inside the scatter kernel).
//
// Per head row x of d bf16 values at global sequence position p:
//     y = x / sqrt(mean(x^2) + eps) * w,   (y[2j], y[2j+1]) rotated by p * theta^(-2j/d),
// in fp32, rounded once to bf16 (nearest even), and written where mode 0 places the row.
//
// Structure: a persistent grid of several CTAs per SM, each with a ring of K shared-memory
// stages. A work unit is a few consecutive tokens of one source rank: all N heads of q and of k,
// two contiguous spans of the sequence-side tensors. A packed input (C planes per token, such as
// the interleaved (b, s, 3, N, d) QKV or QKVG layouts, FastVideo, "Ulysses performance on GB200")
// is cut into blocks of twice as many tokens with C units each (the q and k rows of the first
// half, of the second half, and one unit per other plane with that plane's rows of the whole
// block), so that every unit fills the same stage and the other planes pass through without
// arithmetic. The grid takes every q,k unit first and then each other plane's units in turn: at
// any time it writes 16 destination streams (q, k of 8 ranks) or 8 (one plane), not 24, which
// measured 6.5% faster than rotating through the three kinds of a QKV input. Warp roles per CTA:
//  * loader: lane 0 waits for the stage to be free ("empty" mbarrier), starts the cp.async.bulk
//    loads (completing on the stage's "full" mbarrier as transaction bytes) and leaves a record
//    of the unit beside the stage; while the copies fly, all lanes fill the stage's cos/sin
//    table for the unit's positions and arrive on "full", so a consumer that sees the phase
//    complete sees data, table and record (each unit is decoded once, by the loader);
//  * storer: when the consumers report a unit done ("computed"), the lanes issue one
//    cp.async.bulk store per (token, q|k, destination rank): n_r heads that are contiguous in the
//    stage and in the destination; as soon as those stores have read shared memory (kFusedDrain
//    units later; 0 by default, so right away) the stage is handed back to the loader ("empty");
//  * consumers: one warp takes the q rows, one the k rows. A group of 8 lanes holds one head
//    row (each lane 8 of its RoPE pairs as packed fp32 values, two 16-byte shared-memory
//    accesses per lane; fused_row.cuh) and keeps 3 rows in flight; the sum of squares is reduced
//    with xor shuffles inside the group, the weight and rotation are applied in registers, and
//    the result overwrites its input in shared memory. Each consumer warp then fences its writes
//    for the async proxy and arrives on "computed".
// Measured at the Wan shape, throughput grows with the number of CTAs issuing bulk copies per SM
// more than with ring depth, so the default footprint is small (2 stages of one token's q and k)
// and 4 CTAs share an SM; wider rows fall back to fewer CTAs per SM (see fused_geometry). Two
// consumer warps of 8-lane rows with 3 rows in flight (128 registers a thread) measured faster
// than four of 16-lane rows (80 registers), for both RoPE pair layouts.
//
// RoPE angles: p * theta^(-2j/d) reaches ~75,600 rad at the Wan shape, where an fp32 product
// alone is off by ~5e-3 rad. The angle is formed in turns (units of 2 pi): the host supplies
// theta^(-2j/d) / (2 pi) as a float pair hi + lo; p * hi is split exactly into a product and its
// fma residual (Dekker's error-free product via fma), the whole turns are dropped (exact), the
// small terms are added, and sincospif is called on the reduced fraction. The angle error stays
// near 1e-6 rad.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/ulysses.h"
#include "fused_row.cuh"
#include "plan.h"
#include "ptx.cuh"

namespace uly {

static __device__ unsigned g_fused_status;

#ifndef ULY_FUSED_CTAS_PER_SM
#define ULY_FUSED_CTAS_PER_SM 4
#endif
#ifndef ULY_FUSED_CONSUMER_WARPS
#define ULY_FUSED_CONSUMER_WARPS 2
#endif
#ifndef ULY_FUSED_STAGE_TARGET
#define ULY_FUSED_STAGE_TARGET 20480
#endif
#ifndef ULY_FUSED_MAX_STAGES
#define ULY_FUSED_MAX_STAGES 2
#endif
#ifndef ULY_FUSED_DRAIN
#define ULY_FUSED_DRAIN 0
#endif
constexpr int kFusedCtasPerSm = ULY_FUSED_CTAS_PER_SM;
constexpr int kFusedMaxStages = ULY_FUSED_MAX_STAGES;
constexpr int kFusedDrain = ULY_FUSED_DRAIN;  // store groups left draining when a stage refills
constexpr int kFusedHeader = 256;  // three barriers per stage, then one unit record per stage
constexpr int kFusedRecordsAt = 128;
static_assert(3 * 8 * kFusedMaxStages <= kFusedRecordsAt, "stage barriers must fit the header");
static_assert(kFusedRecordsAt + 16 * kFusedMaxStages <= kFusedHeader, "unit records must fit");
static_assert(kFusedDrain >= 0 && kFusedDrain < kFusedMaxStages, "need a load in flight");
static_assert(ULY_FUSED_CONSUMER_WARPS % 2 == 0, "consumer warps split evenly between q and k");
// warp roles
constexpr int kLoaderWarp = 0, kStorerWarp = 1, kFirstConsumerWarp = 2;
constexpr int kFusedThreads = 32 * (kFirstConsumerWarp + ULY_FUSED_CONSUMER_WARPS);
#ifndef ULY_FUSED_ILP
#define ULY_FUSED_ILP 3
#endif
constexpr int kIlp = ULY_FUSED_ILP;  // head rows in flight per lane group
#ifndef ULY_FUSED_ILP_WIDE  // the same for the 8-pair row layout (rotate half), twice the values
#define ULY_FUSED_ILP_WIDE 3
#endif
constexpr int kIlpWide = ULY_FUSED_ILP_WIDE;
#ifndef ULY_FUSED_WIDE  // 1: 8 RoPE pairs per lane for adjacent pairs too (fused_row.cuh)
#define ULY_FUSED_WIDE 1
#endif
constexpr bool kFusedWide = ULY_FUSED_WIDE != 0;

// What the storer and the consumers need of a unit, written by the loader beside the stage
// before its last arrive on "full" (the loader decodes each unit once).
struct FusedRecord {
    int64_t head_row0;  // first row of the unit on the head side: bb * S + seq_off(q) + i0
    int32_t ntok;
    int32_t kind;       // 0, 1: q and k rows; 2 + 4 c: plane c's rows, moved plain (packed calls)
};

#ifndef ULY_FUSED_WAIT_HINT_NS  // suspend-time hint of the barrier waits (0: plain polling)
#define ULY_FUSED_WAIT_HINT_NS 10000
#endif

__device__ __forceinline__ bool fused_wait(uint64_t* bar, uint32_t parity)
{
#if ULY_FUSED_WAIT_HINT_NS > 0
    return mbar_wait_bounded_hint<ULY_FUSED_WAIT_HINT_NS>(bar, parity);
#else
    return mbar_wait_bounded(bar, parity);
#endif
}

struct FusedUnit {
    int q;
    int64_t bb, i0;
    int ntok;   // may be 0: the second q,k unit of a packed block that holds few tokens
    int kind;   // 0, 1: q and k rows of the block's first / second tokens_per_unit tokens; 2: a
                // plain plane's rows
    int plane;  // kind 2: the plane
};

__device__ __forceinline__ FusedUnit fused_decode(const FusedArgs& a, int64_t u)
{
    FusedUnit t;
    int64_t blk_id = u;
    t.kind = 0;
    t.plane = 0;
    if (a.interleaved) {  // phases: every q,k unit (two per block), then each plain plane's units
        const int64_t blocks_all = a.unit_begin[kMaxW];
        if (u < 2 * blocks_all) {
            blk_id = u >> 1;
            t.kind = int(u & 1);
        } else {
            const int64_t v = u - 2 * blocks_all;
            const int pp = int(div_fast(v, blocks_all));
            blk_id = v - int64_t(pp) * blocks_all;
            t.kind = 2;
            t.plane = a.plain_plane[pp];
        }
    }
    int lo = 0, hi = a.W - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.unit_begin[mid] <= blk_id)
            lo = mid;
        else
            hi = mid - 1;
    }
    t.q = lo;
    const int64_t BT = a.block_tokens;
    const int64_t rows = a.rows[lo];
    const int64_t blocks = a.blocks[lo];  // token blocks per batch index of shard q
    const int64_t local = blk_id - a.unit_begin[lo];
    t.bb = div_fast(local, blocks);
    const int64_t blk = local - t.bb * blocks;
    t.i0 = a.row_lo[lo] + blk * BT;
    const int64_t nblk = min(BT, rows - blk * BT);  // tokens of the block
    const int64_t T = a.tokens_per_unit;
    if (t.kind == 0)
        t.ntok = int(min(T, nblk));
    else if (t.kind == 1) {
        t.i0 += T;
        t.ntok = int(nblk > T ? nblk - T : 0);
    } else {
        t.ntok = int(nblk);
    }
    return t;
}

// Shared-memory layout (byte offsets), shared by the kernel and its launcher.
struct FusedSmem {
    int turns;      // float2 (hi, lo) per pair j < d/2
    int tables;     // per stage: float2 (cos, sin) per (token, pair)
    int stages;     // per stage: q span then k span
    int table_bytes;
    int total;
};

__host__ __device__ inline FusedSmem fused_smem_layout(int d, int tokens, int stages,
                                                       uint32_t stage_bytes)
{
    auto up = [](int x) { return (x + 127) & ~127; };
    FusedSmem m;
    m.turns = kFusedHeader;
    m.tables = up(m.turns + (d / 2) * 8);
    m.table_bytes = up(tokens * (d / 2) * 8);
    m.stages = up(m.tables + stages * m.table_bytes);
    m.total = m.stages + stages * int(stage_bytes);
    return m;
}

// D: head dimension, a power of two, or below 8 for a.d with one of the run-time row layouts
// (rt_layout_for: any multiple of 8 up to 256); F16: fp16 elements (else bf16); HALF_PAIRS:
// rotate-half RoPE pairs (else adjacent pairs). The row layouts (G lanes per row, H packed slots
// per lane) are in fused_row.cuh.
template <int D, bool F16, bool HALF_PAIRS>
__global__ void __launch_bounds__(kFusedThreads, kFusedCtasPerSm)
    fused_qk_kernel(const __grid_constant__ FusedArgs a)
{
    using IO = RowIO<F16, HALF_PAIRS, D, kFusedWide>;
    const int dd = rt_layout(D) ? a.d : D;            // head dimension
    const RowDims dims = IO::dims(dd);
    const int G = dims.g;                  // lanes per head row
    constexpr int H = IO::H;
    const int HALF = dd / 2;
    // lanes from a row's first to the next row's: G, or G rounded up to a power of two
    const int GP = !rt_layout(D) ? G : rt_pow2(D) ? row_lane_stride(G) : G;
    const int GPW = 32 / GP;  // head rows per warp per slot
    // rows in flight per lane group: a lane of an 8-pair layout holds twice the values
    constexpr int ILP = IO::P == 8 ? kIlpWide : kIlp;
    const int PER_STEP = GPW * ILP;
    constexpr int NW = ULY_FUSED_CONSUMER_WARPS;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int K = a.stages;
    const int N = int(a.N);
    const FusedSmem L = fused_smem_layout(dd, a.tokens_per_unit, K, a.stage_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);    // data landed + rope table written
    uint64_t* computed = full + kFusedMaxStages;           // consumers done with the stage
    uint64_t* empty = computed + kFusedMaxStages;          // stores have read the stage
    float2* turns = reinterpret_cast<float2*>(smem + L.turns);
    FusedRecord* records = reinterpret_cast<FusedRecord*>(smem + kFusedRecordsAt);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t first = blockIdx.x, step = gridDim.x;
    const int64_t n = first < a.total_units ? (a.total_units - 1 - first) / step + 1 : 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < K; ++s) {
            mbar_init(&full[s], 1 + 32);  // the loader's expect_tx, then its lanes' table writes
            mbar_init(&computed[s], NW);
            mbar_init(&empty[s], 1);
        }
        fence_barrier_init();
    }
    for (int j = threadIdx.x; j < HALF; j += blockDim.x) turns[j] = make_float2(a.turn_hi[j], a.turn_lo[j]);
    __syncthreads();
    if (n == 0) return;
    const int row_bytes = N * dd * 2;  // one token, all heads, one tensor
    const bool qkv = a.interleaved != 0;
    // Stage layouts. A q,k unit holds row (token t, plane c in {q, k}, head h) at
    // t * tok_stride + c * plane_stride(ntok) + h * 2d: separate inputs arrive as two spans (all q
    // rows, then all k rows), a packed input as one copy per token of its q and k rows (two when
    // the k plane does not follow the q plane). A plain-plane unit (packed only) holds its tokens'
    // rows of that plane back to back, one copy per token.
    const int tok_stride = qkv ? 2 * row_bytes : row_bytes;
    auto plane_stride = [&](int ntok) { return qkv ? row_bytes : ntok * row_bytes; };

    if (warp == kLoaderWarp) {
        // Lane 0 streams units into the stages and leaves each unit's record beside its stage;
        // while the copies fly, the lanes fill the stage's cos/sin table for the unit's positions
        // (free: the stage's previous unit has been stored, so its consumers are done) and
        // arrive on "full", so a consumer that sees the phase complete sees data, table and
        // record.
        int64_t j = 0;
        StageRing ring;
        for (; j < n; ++j, ring.next(K)) {
            const int s = ring.s;
            int ok = 1;
            if (lane == 0 && j >= K) ok = fused_wait(&empty[s], ring.phase ^ 1u);
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                if (lane == 0) atomicOr(&g_fused_status, kStatusWaitTimeout);
                break;
            }
            const FusedUnit t = fused_decode(a, first + j * step);
            const bool v_unit = t.kind == 2;
            const uint32_t bytes = uint32_t(t.ntok) * uint32_t(row_bytes);  // one plane
            const int64_t tok0 = t.bb * a.s[t.q] + t.i0;                      // first source row
            uint8_t* dst = smem + L.stages + size_t(s) * a.stage_bytes;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[s], v_unit ? bytes : 2 * bytes);
                if (!qkv) {
                    bulk_g2s(dst, a.q_in[t.q] + tok0 * row_bytes, bytes, &full[s]);
                    bulk_g2s(dst + bytes, a.k_in[t.q] + tok0 * row_bytes, bytes, &full[s]);
                }
                FusedRecord& rec = records[s];  // published by this lane's arrive below
                rec.head_row0 = t.bb * a.S + a.seq_off[t.q] + t.i0;
                rec.ntok = t.ntok;
                rec.kind = t.kind + 4 * t.plane;
            }
            if (qkv) {  // per token: its q and k rows (one copy when k's plane follows q's), or
                        // its row of the unit's plane
                __syncwarp();  // after lane 0 registered the unit's bytes
                const uint8_t* src = a.packed_in[t.q] + tok0 * a.tok_pitch;
                if (v_unit) {
                    const uint8_t* from = src + int64_t(t.plane) * row_bytes;
                    for (int tok = lane; tok < t.ntok; tok += 32)
                        bulk_g2s(dst + size_t(tok) * row_bytes, from + int64_t(tok) * a.tok_pitch,
                                 uint32_t(row_bytes), &full[s]);
                } else if (a.k_plane == a.q_plane + 1) {
                    const uint8_t* from = src + int64_t(a.q_plane) * row_bytes;
                    for (int tok = lane; tok < t.ntok; tok += 32)
                        bulk_g2s(dst + size_t(tok) * 2 * row_bytes, from + int64_t(tok) * a.tok_pitch,
                                 2u * uint32_t(row_bytes), &full[s]);
                } else {
                    for (int c = lane; c < 2 * t.ntok; c += 32) {
                        const int tok = c >> 1, which = c & 1;
                        const int plane = which ? a.k_plane : a.q_plane;
                        bulk_g2s(dst + size_t(c) * row_bytes,
                                 src + int64_t(tok) * a.tok_pitch + int64_t(plane) * row_bytes,
                                 uint32_t(row_bytes), &full[s]);
                    }
                }
            }
            float* table = reinterpret_cast<float*>(smem + L.tables + s * L.table_bytes);
            const float p0 = float(a.seq_off[t.q] + t.i0);
            // Per token, lane i of a row group owns pairs P i .. P i + P - 1, read as P / 2
            // 16-byte entries (c_j, c_j+1, s_j, s_j+1) for j = P i + 2h; for each h the entries
            // of all lanes are adjacent, so each read is contiguous.
            for (int e = lane; e < (v_unit ? 0 : t.ntok * HALF); e += 32) {
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
                    atomicOr(&g_fused_status, kStatusDrainTimeout);
                    break;
                }
            }
        }
        return;
    }

    if (warp == kStorerWarp) {
        // The results sit where their inputs were (v rows untouched): for each token, plane and
        // destination rank one run of n_r heads, contiguous in the stage and in the destination
        // tensor. A stage is handed back to the loader kFusedDrain units later, once its stores
        // have read it.
        int64_t j = 0;
        StageRing ring;
        for (; j < n; ++j, ring.next(K)) {
            const int s = ring.s;
            if (!__all_sync(0xffffffffu, fused_wait(&computed[s], ring.phase))) {
                if (lane == 0) atomicOr(&g_fused_status, kStatusWaitTimeout);
                break;
            }
            const FusedRecord rec = records[s];
            const uint8_t* st = smem + L.stages + size_t(s) * a.stage_bytes;
            const int64_t row0 = rec.head_row0;
            const int W = a.W;
            const bool v_unit = (rec.kind & 3) == 2;
            uint8_t* const* plain_out = a.plane_out[rec.kind >> 2];
            const int uplanes = v_unit ? 1 : 2;
            const int ustride = v_unit ? row_bytes : tok_stride;
            const int pstride = plane_stride(rec.ntok);
            const int runs = rec.ntok * uplanes * W;
            for (int idx = lane; idx < runs; idx += 32) {
                const int rest = idx / W, r = idx - rest * W;
                const int tok = rest / uplanes, plane = rest - tok * uplanes;
                const int64_t run = a.n[r] * (dd * 2);
                if (run == 0) continue;
                const uint8_t* src = st + tok * ustride + plane * pstride + a.head_off[r] * (dd * 2);
                uint8_t* out = v_unit ? plain_out[r] : plane == 0 ? a.q_out[r] : a.k_out[r];
                bulk_s2g(out + (row0 + tok) * run, src, uint32_t(run));
            }
            bulk_commit();
            if (j >= kFusedDrain) {
                bulk_wait_read<kFusedDrain>();  // unit j - kFusedDrain has left shared memory
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[(j - kFusedDrain) % K]);
            }
        }
        bulk_wait<0>();
        return;
    }

    // consumers: the first half of the warps normalise q rows, the second half k rows
    constexpr int HALF_NW = NW / 2;
    const int cw = warp - kFirstConsumerWarp;
    const int which = cw >= HALF_NW;          // 0: q, 1: k (uniform per warp)
    const int cwi = cw - which * HALF_NW;     // rank among the warps of this tensor
    const int group = lane / GP;       // which head row of the warp slot
    const int sub = lane - group * GP;  // which pairs of the row this lane holds
    const bool active = sub < G && group < GPW;  // lanes holding no row's pairs (run-time d)
    // This lane's weights as packed pairs: first / second elements of its pairs, plus the
    // negated second ones (the rotation subtracts them).
    float2 wE[H], wO[H], wOn[H];
    for (int h = 0; h < H; ++h) wE[h] = wO[h] = make_float2(0.f, 0.f);
    if (active) IO::weights(a.rms_w + which * dd, sub, wE, wO, dims);
    for (int h = 0; h < H; ++h) wOn[h] = make_float2(-wO[h].x, -wO[h].y);
    const float inv_d = 1.0f / float(dd);
    // this warp's share of the rows of a full token block (steps m_lo .. m_hi - 1 of PER_STEP
    // rows) and the (token, head) of its first row
    const int full_steps = (a.tokens_per_unit * N + PER_STEP - 1) / PER_STEP;
    const int full_m_lo = cwi * full_steps / HALF_NW, full_m_hi = (cwi + 1) * full_steps / HALF_NW;
    const int full_base_tok = full_m_lo * PER_STEP / N;
    const int full_base_head = full_m_lo * PER_STEP - full_base_tok * N;
    StageRing ring;
    for (int64_t k = 0; k < n; ++k, ring.next(K)) {
        const int s = ring.s;
        if (!__all_sync(0xffffffffu, fused_wait(&full[s], ring.phase))) {
            if (lane == 0) atomicOr(&g_fused_status, kStatusWaitTimeout);
            break;
        }
        if ((records[s].kind & 3) == 2) {  // a plain plane's rows: nothing to compute
            __syncwarp();
            if (lane == 0) mbar_arrive(&computed[s]);
            continue;
        }
        const int ntok = records[s].ntok;
        // this tensor's plane in the stage; row (token, head) at token * tok_stride + head * 2d
        uint8_t* rows_base = smem + L.stages + size_t(s) * a.stage_bytes + which * plane_stride(ntok);
        const float4* table = reinterpret_cast<const float4*>(smem + L.tables + s * L.table_bytes);
        const int rows = ntok * N;
        int m_lo = full_m_lo, m_hi = full_m_hi;
        int base_tok = full_base_tok, base_head = full_base_head;
        if (ntok != a.tokens_per_unit) {  // a short block: this warp's share of its rows
            const int steps = (rows + PER_STEP - 1) / PER_STEP;
            m_lo = cwi * steps / HALF_NW;
            m_hi = (cwi + 1) * steps / HALF_NW;
            base_tok = m_lo * PER_STEP / N;
            base_head = m_lo * PER_STEP - base_tok * N;
        }
        int base = m_lo * PER_STEP;   // first row of the current step and its (token, head)
        for (int m = m_lo; m < m_hi; ++m) {
            uint8_t* slot[ILP];
            int tok[ILP];
            bool ok[ILP];
            // first / second elements of this lane's pairs, packed
            float2 vE[ILP][H], vO[ILP][H];
            float ss[ILP];
#pragma unroll
            for (int u = 0; u < ILP; ++u) {
                const int o = u * GPW + group;
                ok[u] = base + o < rows;
                int hh = base_head + o, tk = base_tok;
                while (hh >= N) {
                    hh -= N;
                    ++tk;
                }
                slot[u] = rows_base + tk * tok_stride + hh * (dd * 2);
                tok[u] = tk;
                typename IO::Words x = {};
                if (ok[u] && active) x = IO::load(slot[u], sub, dims);
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    IO::unpack(x, h, vE[u][h], vO[u][h]);
                    acc = __ffma2_rn(vE[u][h], vE[u][h], acc);
                    acc = __ffma2_rn(vO[u][h], vO[u][h], acc);
                }
                ss[u] = acc.x + acc.y;
            }
            row_sums<D, 1>(ss, ss, G, GP, sub, group);
#pragma unroll
            for (int u = 0; u < ILP; ++u) {
                if (!ok[u] || !active) continue;
                const float inv = rsqrtf(ss[u] * inv_d + a.eps);
                const float2 inv2 = make_float2(inv, inv);
                float2 oEs[H], oOs[H];
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    // (c_j, c_j+1, s_j, s_j+1) for j = P sub + 2 h (see the table layout)
                    const float4 cs = table[IO::table_entry(tok[u], h, sub, dims)];
                    const float2 c2 = make_float2(cs.x, cs.y), s2 = make_float2(cs.z, cs.w);
                    const float2 A = __fmul2_rn(vE[u][h], wE[h]);   // weighted first elements
                    const float2 Bp = __fmul2_rn(vO[u][h], wO[h]);  // weighted second elements
                    const float2 Bn = __fmul2_rn(vO[u][h], wOn[h]);
                    // rotation, then the 1/rms factor (the rotation is linear)
                    oEs[h] = __fmul2_rn(__ffma2_rn(Bn, s2, __fmul2_rn(A, c2)), inv2);
                    oOs[h] = __fmul2_rn(__ffma2_rn(A, s2, __fmul2_rn(Bp, c2)), inv2);
                }
                IO::store(slot[u], sub, IO::pack(oEs, oOs), dims);  // in place
            }
            base += PER_STEP;
            base_head += PER_STEP;
            while (base_head >= N) {
                base_head -= N;
                ++base_tok;
            }
        }
        // make this warp's shared-memory results visible to the bulk-copy unit, then report
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) mbar_arrive(&computed[s]);
    }
}

// Stage geometry for a plan: tokens per unit and stage count (0 stages: does not fit).
// Stage geometry for a plan: tokens per unit, stage count and CTAs per SM (0 stages: one
// token's q and k rows do not fit even one CTA per SM). The preferred footprint lets
// kFusedCtasPerSm CTAs share an SM; narrower units, fewer stages, then fewer CTAs per SM are
// tried in that order.
void fused_geometry(const Plan& p, int planes, int64_t* tokens_per_unit, int* stages,
                    uint32_t* stage_bytes, int* ctas_per_sm)
{
    *stages = 0;
    *tokens_per_unit = 1;
    *stage_bytes = 0;
    *ctas_per_sm = 1;
    const int64_t pair_bytes = planes * p.N * p.d * 2;  // one token of q and k (and v)
    int64_t T0 = ULY_FUSED_STAGE_TARGET / pair_bytes;
    if (T0 < 1) T0 = 1;
    const int min_k = kFusedDrain + 1 > 2 ? kFusedDrain + 1 : 2;
    for (int ctas = kFusedCtasPerSm; ctas >= 1; --ctas) {
        const int budget = kSmemPerSm / ctas - kSmemReservedPerCta;
        for (int64_t T = T0; T >= 1; T = T > 1 ? T / 2 : 0) {
            const int64_t sb = T * pair_bytes;
            if (sb > (1 << 20)) continue;
            for (int K = kFusedMaxStages; K >= min_k; --K) {
                const FusedSmem m = fused_smem_layout(int(p.d), int(T), K, uint32_t(sb));
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

template <int D, bool F16, bool HALF>
static cudaError_t launch_d(const FusedArgs& a, cudaStream_t stream, int device, int grid)
{
    static std::atomic<unsigned long long> raised{0};  // devices with this variant's limit raised
    const unsigned long long bit = device >= 0 && device < 64 ? 1ull << device : 0;
    if (bit && !(raised.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(fused_qk_kernel<D, F16, HALF>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemPerCtaMax);
        if (e != cudaSuccess) return e;
        raised.fetch_or(bit);
    }
    const FusedSmem m = fused_smem_layout(a.d, a.tokens_per_unit, a.stages, a.stage_bytes);
    fused_qk_kernel<D, F16, HALF><<<grid, kFusedThreads, m.total, stream>>>(a);
    return cudaGetLastError();
}

template <int D>
static cudaError_t launch_variant(const FusedArgs& a, cudaStream_t stream, int device, int grid)
{
    if (a.elem_f16)
        return a.rope_half ? launch_d<D, true, true>(a, stream, device, grid)
                           : launch_d<D, true, false>(a, stream, device, grid);
    return a.rope_half ? launch_d<D, false, true>(a, stream, device, grid)
                       : launch_d<D, false, false>(a, stream, device, grid);
}

cudaError_t fused_launch(const FusedArgs& a, cudaStream_t stream, int device, int sm_count,
                         int64_t max_grid)
{
    if (a.total_units == 0) return cudaSuccess;
    int64_t grid = int64_t(sm_count) * (a.ctas_per_sm > 0 ? a.ctas_per_sm : 1);
    if (max_grid > 0 && grid > max_grid) grid = max_grid;
    if (grid > a.total_units) grid = a.total_units;
    switch (a.d) {
        case 8: return launch_variant<8>(a, stream, device, int(grid));
        case 16: return launch_variant<16>(a, stream, device, int(grid));
        case 32: return launch_variant<32>(a, stream, device, int(grid));
        case 64: return launch_variant<64>(a, stream, device, int(grid));
        case 128: return launch_variant<128>(a, stream, device, int(grid));
        case 256: return launch_variant<256>(a, stream, device, int(grid));
        default:  // any other multiple of 8 up to 256: a run-time row layout
            if (a.d % 8 != 0 || a.d < 8 || a.d > kMaxFusedD) return cudaErrorInvalidValue;
            switch (rt_layout_for(a.d)) {
                case 0: return launch_variant<0>(a, stream, device, int(grid));
                case kRtWide: return launch_variant<kRtWide>(a, stream, device, int(grid));
                case kRtPow2: return launch_variant<kRtPow2>(a, stream, device, int(grid));
                default: return launch_variant<kRtPow2 | kRtWide>(a, stream, device, int(grid));
            }
    }
}

cudaError_t fused_status(unsigned* status, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(status, g_fused_status, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_fused_status, &zero, sizeof(unsigned));
}

}  // namespace uly
