// fused_qk_tensor.cu -- the fused QK call (mode-0 relayout of q and k with QK RMSNorm + RoPE in the
// scatter; fast-ulysses 0.1.0, "Fusion examples") with row-block units reordered by a tensor map.
//
// The arithmetic is the token-unit kernel's (fused_qk.cu): per head row x of d values at global
// sequence position p, y = x / sqrt(mean(x^2) + eps) * w, pairs rotated by p * theta^(-2j/d), in
// fp32, rounded once. What differs is how rows move. A unit is a block of R consecutive rows of
// one sequence shard and batch index, all N heads, of q and of k. Each tensor's block arrives with
// ONE tiled tensor-map copy whose map walks the heads as (run, row, head group): the box lands in
// shared memory group-major, [group][row][run], so each destination rank's rows of the block are
// already back to back, as its head-side tensor holds them. After the consumers normalise and
// rotate in place, each (tensor, rank) leaves with one contiguous bulk store of R runs. Per unit
// 2 copies in and 2 W out, for R tokens (the token-unit kernel: 2 in and 2 W out per token).
// It needs every head group's run (n d e bytes) equal and at most 2,048 bytes (the box's inner
// extent); other plans use the token units.
//
// Packed inputs (C planes per token at a token pitch, such as the interleaved (b, s, 3, N, d) QKV
// or QKVG layouts; FastVideo, "Ulysses performance on GB200") take the same maps with the token
// pitch as their row stride. Their other planes move without arithmetic in units of 2R rows of
// one plane (one box of the same bytes as a q,k unit): one copy in, W out. The grid takes every
// q,k unit first, then each other plane's units in turn.
//
// Warp roles per CTA: a loader (lane 0 issues the two tensor loads and leaves the unit's record),
// a storer (one lane per (tensor, rank) store, once the consumers are done; the stage goes back to
// the loader when the stores have read it), and consumer warps, half on q rows and half on k rows,
// with the token-unit kernel's row layout (fused_row.cuh: 8 lanes per head row, packed fp32x2
// arithmetic). The consumers also fill the unit's cos/sin table, shared out among them while the
// unit's copies are in flight, and meet at a named barrier before using it. Every wait is bounded.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>

#include "../../include/ulysses.h"
#include "fused_row.cuh"
#include "plan.h"
#include "ptx.cuh"
#include "tensor_map.h"

namespace uly {

static __device__ unsigned g_fused_tensor_status;

#ifndef ULY_FT_BOX_BYTES  // target bytes of one tensor's box (R whole rows) ...
#define ULY_FT_BOX_BYTES 24576
#endif
#ifndef ULY_FT_MIN_ROWS  // ... but at least this many rows
#define ULY_FT_MIN_ROWS 3
#endif
#ifndef ULY_FT_STAGES
#define ULY_FT_STAGES 3
#endif
#ifndef ULY_FT_CTAS_PER_SM
#define ULY_FT_CTAS_PER_SM 1
#endif
#ifndef ULY_FT_CONSUMER_WARPS
#define ULY_FT_CONSUMER_WARPS 16
#endif
#ifndef ULY_FT_ILP  // head rows in flight per lane group
#define ULY_FT_ILP 1
#endif
constexpr int kFtStages = ULY_FT_STAGES;
constexpr int kFtConsumerWarps = ULY_FT_CONSUMER_WARPS;
constexpr int kFtThreads = 32 * (2 + kFtConsumerWarps);
constexpr int kFtRecordsAt = 128;  // barriers first, then one unit record per stage
constexpr int kFtTurnsAt = 256;
constexpr int kFtTableBarrier = 1;  // named barrier of the consumer warps (0 is __syncthreads)
static_assert(3 * 8 * kFtStages <= kFtRecordsAt, "stage barriers must fit the header");
static_assert(kFtRecordsAt + 16 * kFtStages <= kFtTurnsAt, "unit records must fit the header");
static_assert(kFtConsumerWarps % 2 == 0, "consumer warps split evenly between q and k");

constexpr int kMaxPlain = kMaxPlanes - 2;  // planes of a packed input other than q and k

struct FusedTensorArgs {
    CUtensorMap qmap[kMaxW];  // per source shard: (run / 8, rows, W, b), see encode_group_map
    CUtensorMap kmap[kMaxW];
    CUtensorMap pmap[kMaxPlain][kMaxW];  // packed inputs: the other planes, boxes of 2R rows
    uint8_t* q_out[kMaxW];
    uint8_t* k_out[kMaxW];
    uint8_t* plain_out[kMaxPlain][kMaxW];
    const float* rms_w;  // [2][d]
    int64_t seq_off[kMaxW];
    int64_t row_lo[kMaxW], rows[kMaxW];  // this launch's rows of shard q
    int64_t blocks[kMaxW];               // q,k units: blocks of R rows per batch index of shard q
    int64_t unit_begin[kMaxW + 1];       // prefix of q,k unit counts over q
    int64_t blocks2[kMaxW];              // other planes: blocks of 2R rows per batch index
    int64_t unit_begin2[kMaxW + 1];      // prefix of one plane's unit counts over q
    int64_t S, R, total_units;
    int64_t qk_units;     // units 0 .. qk_units - 1 are q,k units; then n_plain phases of
    int64_t plain_units;  // plain_units each
    int32_t n_plain;
    int32_t W, n;         // ranks; heads per rank (every rank the same)
    int32_t d;            // head dimension
    uint32_t run;         // n * d * elem_size: bytes of one rank's part of a row
    uint32_t box_bytes;   // R * W * run: one tensor's box
    uint32_t box_stride;  // bytes from a stage's q box to its k box (a multiple of 128)
    uint32_t stage_bytes;
    uint32_t table_bytes;  // one stage's cos/sin table: R rows x d/2 pairs x 8 bytes
    float eps;
    float turn_hi[kMaxFusedD / 2];  // theta^(-2j/d) / (2 pi) as hi + lo, j < d/2
    float turn_lo[kMaxFusedD / 2];
};

struct FtRecord {
    int64_t head_row0;  // the unit's first row on the head side: bb * S + seq_off(q) + row
    int32_t nrows;
    int32_t kind;       // 0: q and k rows; 1 + p: other plane p's rows, moved plain
};

struct FtUnit {
    int q, kind;
    int64_t bb, i0, nrows;  // i0: first row in this launch's rows of shard q
};

__device__ __forceinline__ FtUnit ft_decode(const FusedTensorArgs& a, int64_t u)
{
    FtUnit t;
    t.kind = 0;
    const int64_t* begin = a.unit_begin;
    const int64_t* blocks_of = a.blocks;
    int64_t R = a.R;
    if (u >= a.qk_units) {  // another plane's unit: blocks of 2R rows
        const int64_t v = u - a.qk_units;
        const int64_t p = div_fast(v, a.plain_units);
        t.kind = int(1 + p);
        u = v - p * a.plain_units;
        begin = a.unit_begin2;
        blocks_of = a.blocks2;
        R *= 2;
    }
    int lo = 0, hi = a.W - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (begin[mid] <= u)
            lo = mid;
        else
            hi = mid - 1;
    }
    t.q = lo;
    const int64_t local = u - begin[lo];
    const int64_t blocks = blocks_of[lo];
    t.bb = div_fast(local, blocks);
    t.i0 = (local - t.bb * blocks) * R;
    t.nrows = min(R, a.rows[lo] - t.i0);
    return t;
}

// Shared-memory layout (byte offsets), shared by the kernel and its launcher.
struct FtSmem {
    int turns, tables, stages, total;
};

__host__ __device__ inline FtSmem ft_smem_layout(int d, uint32_t table_bytes, uint32_t stage_bytes)
{
    auto up = [](int x, int a) { return (x + a - 1) / a * a; };
    FtSmem m;
    m.turns = kFtTurnsAt;
    m.tables = up(m.turns + (d / 2) * 8, 128);
    m.stages = up(m.tables + kFtStages * int(table_bytes), 1024);
    m.total = m.stages + kFtStages * int(stage_bytes);
    return m;
}

__device__ __forceinline__ bool ft_wait(uint64_t* bar, uint32_t parity)
{
    return mbar_wait_bounded_hint<10000>(bar, parity);
}

// D: head dimension, a power of two, or below 8 for a.d with one of the run-time row layouts of
// fused_row.cuh (rt_layout_for: any multiple of 8 up to 256); F16: fp16 elements (else bf16);
// HALF_PAIRS: rotate-half RoPE pairs.
template <int D, bool F16, bool HALF_PAIRS>
__global__ void __launch_bounds__(kFtThreads, ULY_FT_CTAS_PER_SM)
    fused_qk_tensor_kernel(const __grid_constant__ FusedTensorArgs a)
{
    using IO = RowIO<F16, HALF_PAIRS, D, true>;
    const int dd = rt_layout(D) ? a.d : D;  // head dimension
    const RowDims dims = IO::dims(dd);
    const int G = dims.g;        // lanes per head row
    constexpr int H = IO::H;
    const int HALF = dd / 2;
    // lanes from a row's first to the next row's: G, or G rounded up to a power of two
    const int GP = !rt_layout(D) ? G : rt_pow2(D) ? row_lane_stride(G) : G;
    const int GPW = 32 / GP;  // head rows per warp per slot
    constexpr int ILP = ULY_FT_ILP;
    const int PER_STEP = GPW * ILP;
    constexpr int K = kFtStages;
    constexpr int NW = kFtConsumerWarps;
    extern __shared__ __align__(1024) uint8_t smem[];
    const FtSmem L = ft_smem_layout(dd, a.table_bytes, a.stage_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);  // both boxes landed
    uint64_t* computed = full + K;                       // consumers done with the stage
    uint64_t* empty = computed + K;                      // the stores have read the stage
    FtRecord* records = reinterpret_cast<FtRecord*>(smem + kFtRecordsAt);
    float2* turns = reinterpret_cast<float2*>(smem + L.turns);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t first = blockIdx.x, step = gridDim.x;
    const int64_t n = first < a.total_units ? (a.total_units - 1 - first) / step + 1 : 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < K; ++s) {
            mbar_init(&full[s], 1);  // the loader's expect_tx
            mbar_init(&computed[s], NW);
            mbar_init(&empty[s], 1);
        }
        fence_barrier_init();
    }
    for (int j = threadIdx.x; j < HALF; j += blockDim.x)
        turns[j] = make_float2(a.turn_hi[j], a.turn_lo[j]);
    __syncthreads();
    if (n == 0) return;

    if (warp == 0) {  // loader
        int64_t j = 0;
        StageRing ring;
        for (; j < n; ++j, ring.next(K)) {
            const int s = ring.s;
            int ok = 1;
            if (lane == 0 && j >= K) ok = ft_wait(&empty[s], ring.phase ^ 1u);
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                if (lane == 0) atomicOr(&g_fused_tensor_status, kStatusWaitTimeout);
                break;
            }
            if (lane == 0) {
                const FtUnit t = ft_decode(a, first + j * step);
                uint8_t* dst = smem + L.stages + size_t(s) * a.stage_bytes;
                // the whole boxes arrive: rows past the chunk are filled
                mbar_arrive_expect_tx(&full[s], 2 * a.box_bytes);
                if (t.kind == 0) {
                    tensor_g2s_4d(dst, &a.qmap[t.q], 0, int(t.i0), 0, int(t.bb), &full[s]);
                    tensor_g2s_4d(dst + a.box_stride, &a.kmap[t.q], 0, int(t.i0), 0, int(t.bb),
                                  &full[s]);
                } else {  // one box of 2R rows, the same bytes
                    tensor_g2s_4d(dst, &a.pmap[t.kind - 1][t.q], 0, int(t.i0), 0, int(t.bb),
                                  &full[s]);
                }
                FtRecord& rec = records[s];  // published by this lane's arrive
                rec.head_row0 = t.bb * a.S + a.seq_off[t.q] + a.row_lo[t.q] + t.i0;
                rec.nrows = int(t.nrows);
                rec.kind = t.kind;
            }
            __syncwarp();
        }
        // do not leave while copies into this CTA's shared memory may be in flight
        if (lane == 0) {
            for (int64_t jj = (j > K ? j - K : 0); jj < j; ++jj) {
                if (!mbar_wait_bounded(&full[jj % K], uint32_t((jj / K) & 1))) {
                    atomicOr(&g_fused_tensor_status, kStatusDrainTimeout);
                    break;
                }
            }
        }
        return;
    }

    if (warp == 1) {  // storer: lane c < 2 W stores tensor c / W's rows for rank c % W (a q,k
                      // unit), or lane r < W rank r's rows (another plane's unit)
        StageRing ring;
        for (int64_t j = 0; j < n; ++j, ring.next(K)) {
            const int s = ring.s;
            if (!__all_sync(0xffffffffu, ft_wait(&computed[s], ring.phase))) {
                if (lane == 0) atomicOr(&g_fused_tensor_status, kStatusWaitTimeout);
                break;
            }
            const FtRecord rec = records[s];
            const uint8_t* st = smem + L.stages + size_t(s) * a.stage_bytes;
            if (rec.kind == 0 && lane < 2 * a.W) {
                const int t = lane >= a.W, r = lane - t * a.W;
                const uint8_t* src = st + t * a.box_stride + size_t(r) * a.R * a.run;
                uint8_t* dst = (t ? a.k_out[r] : a.q_out[r]) + rec.head_row0 * a.run;
                bulk_s2g(dst, src, uint32_t(rec.nrows) * a.run);
                bulk_commit();
                bulk_wait_read<0>();
            } else if (rec.kind > 0 && lane < a.W) {
                const uint8_t* src = st + size_t(lane) * 2 * a.R * a.run;
                uint8_t* dst = a.plain_out[rec.kind - 1][lane] + rec.head_row0 * a.run;
                bulk_s2g(dst, src, uint32_t(rec.nrows) * a.run);
                bulk_commit();
                bulk_wait_read<0>();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        bulk_wait<0>();
        return;
    }

    // consumers: the first half of the warps normalise q rows, the second half k rows
    constexpr int HALF_NW = NW / 2;
    const int cw = warp - 2;
    const int which = cw >= HALF_NW;       // 0: q, 1: k (uniform per warp)
    const int cwi = cw - which * HALF_NW;  // rank among the warps of this tensor
    const int group = lane / GP;       // which head row of the warp slot
    const int sub = lane - group * GP;  // which pairs of the row this lane holds
    const bool active = sub < G && group < GPW;  // lanes holding no row's pairs (run-time d)
    float2 wE[H], wO[H], wOn[H];
    for (int h = 0; h < H; ++h) wE[h] = wO[h] = make_float2(0.f, 0.f);
    if (active) IO::weights(a.rms_w + which * dd, sub, wE, wO, dims);
    for (int h = 0; h < H; ++h) wOn[h] = make_float2(-wO[h].x, -wO[h].y);
    const float inv_d = 1.0f / float(dd);
    const int ctid = cw * 32 + lane;  // rank among the consumer threads
    const int nr = a.n, R = int(a.R), W = a.W;
    const int run = int(a.run);
    // A box's head rows in order: (group g, row i, head h) at ((g R + i) n + h); this warp's
    // share of the steps of PER_STEP rows, the same for every unit (short units skip the rows
    // past their end).
    const int box_rows = W * R * nr;
    const int steps = (box_rows + PER_STEP - 1) / PER_STEP;
    const int m_lo = cwi * steps / HALF_NW, m_hi = (cwi + 1) * steps / HALF_NW;
    const int start = m_lo * PER_STEP;
    const int start_pt = start / nr;  // pseudo-token g R + i of the first row, and its head
    const int start_head = start - start_pt * nr;
    const int start_g = start_pt / R, start_i = start_pt - start_g * R;
    // Every consumer warp passes the per-unit barrier n times: a warp whose wait timed out keeps
    // going round with its waits and work skipped (the status word records it), so the others
    // never wait at the barrier for a warp that has left.
    bool failed = false;
    StageRing ring;
    for (int64_t k = 0; k < n; ++k, ring.next(K)) {
        const int s = ring.s;
        // The unit's cos/sin table, shared out over the consumer threads while its copies fly:
        // rows i0 .. i0 + nrows - 1 sit at global positions p0 + i. The slot was last read for
        // unit k - K, which every consumer warp finished before the barrier of unit k - 1.
        const FtUnit t = ft_decode(a, first + k * step);
        const int nrows = t.kind == 0 ? int(t.nrows) : 0;  // another plane's unit: no table
        {
            float* table = reinterpret_cast<float*>(smem + L.tables + s * a.table_bytes);
            const float p0 = float(a.seq_off[t.q] + a.row_lo[t.q] + t.i0);
            for (int e = ctid; e < nrows * HALF; e += NW * 32) {
                const int tok = e / HALF, jj = e - tok * HALF;
                const float2 tj = turns[jj];
                const float2 cs = rope_cos_sin(p0 + float(tok), tj.x, tj.y);
                const int at = IO::table_at(tok, jj, dims);
                table[at] = cs.x;
                table[at + 2] = cs.y;
            }
        }
        asm volatile("bar.sync %0, %1;" ::"r"(kFtTableBarrier), "r"(NW * 32) : "memory");
        if (!failed && !__all_sync(0xffffffffu, ft_wait(&full[s], ring.phase))) {
            if (lane == 0) atomicOr(&g_fused_tensor_status, kStatusWaitTimeout);
            failed = true;
        }
        if (failed || t.kind != 0) {  // nothing to compute
            __syncwarp();
            if (lane == 0) mbar_arrive(&computed[s]);
            continue;
        }
        uint8_t* rows_base = smem + L.stages + size_t(s) * a.stage_bytes + which * a.box_stride;
        const float4* table = reinterpret_cast<const float4*>(smem + L.tables + s * a.table_bytes);
        int bg = start_g, bi = start_i, bh = start_head;  // (group, row, head) of the step's first row
        for (int m = m_lo; m < m_hi; ++m) {
            uint8_t* slot[ILP];
            int tok[ILP];
            bool ok[ILP];
            float2 vE[ILP][H], vO[ILP][H];
            float ss[ILP];
#pragma unroll
            for (int u = 0; u < ILP; ++u) {
                int hh = bh + u * GPW + group, ii = bi, gg = bg;
                while (hh >= nr) {
                    hh -= nr;
                    if (++ii == R) {
                        ii = 0;
                        ++gg;
                    }
                }
                ok[u] = gg < W && ii < nrows;
                slot[u] = rows_base + (gg * R + ii) * run + hh * (dd * 2);
                tok[u] = ii;
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
                    const float4 cs = table[IO::table_entry(tok[u], h, sub, dims)];
                    const float2 c2 = make_float2(cs.x, cs.y), s2 = make_float2(cs.z, cs.w);
                    const float2 A = __fmul2_rn(vE[u][h], wE[h]);
                    const float2 Bp = __fmul2_rn(vO[u][h], wO[h]);
                    const float2 Bn = __fmul2_rn(vO[u][h], wOn[h]);
                    oEs[h] = __fmul2_rn(__ffma2_rn(Bn, s2, __fmul2_rn(A, c2)), inv2);
                    oOs[h] = __fmul2_rn(__ffma2_rn(A, s2, __fmul2_rn(Bp, c2)), inv2);
                }
                IO::store(slot[u], sub, IO::pack(oEs, oOs), dims);  // in place
            }
            bh += PER_STEP;
            while (bh >= nr) {
                bh -= nr;
                if (++bi == R) {
                    bi = 0;
                    ++bg;
                }
            }
        }
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) mbar_arrive(&computed[s]);
    }
}

// Whether this kernel takes the plan: every head group's run the same length, at most 2,048
// bytes (the tensor box's inner extent), and no empty group.
bool fused_tensor_fits(const Plan& p)
{
    const int64_t run = p.n[0] * p.d * p.e;
    if (run == 0 || run > 2048) return false;
    for (int r = 1; r < p.W; ++r)
        if (p.n[r] != p.n[0]) return false;
    return true;
}

// The automatic choice between this kernel and the token units. Measured (CUDA events, back to
// back, 75,600-token plans): this kernel's time per byte depends mostly on its stage size, best
// at 48-60 KiB (3 stages), i.e. R = max(3, 24 KiB / row) rows; where three rows of q and k take
// at most 60 KiB (rows of N d e <= 10,240 bytes) it ran at 0.94-1.02 of the copy peak against
// the token units' 0.83-0.98, and with longer rows (fewer than 3 rows per box) below them.
bool fused_tensor_preferred(const Plan& p)
{
    // head dimensions that are not powers of two (the run-time row layouts): the token units
    // measured as fast or faster (d = 72, 80, 96, 120 at 75,600 tokens: 0.67-0.72 against
    // 0.48-0.72 of the copy peak)
    if ((p.d & (p.d - 1)) != 0) return false;
    return fused_tensor_fits(p) && p.N * p.d * p.e <= 10240;
}

template <int D, bool F16, bool HALF>
static cudaError_t ft_launch_d(const FusedTensorArgs& a, int smem, cudaStream_t stream, int device,
                               int grid)
{
    static std::atomic<unsigned long long> raised{0};  // devices with this variant's limit raised
    const unsigned long long bit = device >= 0 && device < 64 ? 1ull << device : 0;
    if (bit && !(raised.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(fused_qk_tensor_kernel<D, F16, HALF>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemPerCtaMax);
        if (e != cudaSuccess) return e;
        raised.fetch_or(bit);
    }
    fused_qk_tensor_kernel<D, F16, HALF><<<grid, kFtThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

template <int D>
static cudaError_t ft_launch_variant(const FusedTensorArgs& a, bool f16, bool half, int smem,
                                     cudaStream_t stream, int device, int grid)
{
    if (f16)
        return half ? ft_launch_d<D, true, true>(a, smem, stream, device, grid)
                    : ft_launch_d<D, true, false>(a, smem, stream, device, grid);
    return half ? ft_launch_d<D, false, true>(a, smem, stream, device, grid)
                : ft_launch_d<D, false, false>(a, smem, stream, device, grid);
}

// One launch over the given rows of every shard (the plan must fit: fused_tensor_fits). `f`
// holds the call's checked pointers, weights, eps and RoPE turns (fused_prepare).
cudaError_t fused_tensor_launch(const Plan& p, const FusedArgs& f, const ChunkRows& rows,
                                cudaStream_t stream, int device, int sm_count, int64_t max_grid)
{
    FusedTensorArgs a;
    std::memset(&a, 0, sizeof a);
    const int W = p.W;
    const int64_t de = p.d * p.e;
    const int64_t run = p.n[0] * de;
    const int64_t row = W * run;  // N * d * e
    const bool packed = f.interleaved != 0;
    const int n_plain = packed ? f.planes - 2 : 0;
    const int64_t pitch = packed ? f.tok_pitch : row;  // bytes from one token to the next
    a.R = ULY_FT_BOX_BYTES / row;
    if (a.R < ULY_FT_MIN_ROWS) a.R = ULY_FT_MIN_ROWS;
    if (a.R > 128) a.R = 128;  // a box holds at most 256 rows: 2R for the other planes
    if (a.R < 1) a.R = 1;
    auto up = [](int64_t x, int64_t m) { return (x + m - 1) / m * m; };
    auto fits = [&](int64_t R) {  // R rows' stages fit one CTA's shared memory
        const uint32_t box = uint32_t(up(R * row, 128));
        const uint32_t table = uint32_t(up(R * (p.d / 2) * 8, 128));
        return ft_smem_layout(int(p.d), table, 2 * box).total <= kSmemPerCtaMax;
    };
    while (!fits(a.R)) {  // the largest block of rows whose stages fit
        if (a.R == 1) return cudaErrorInvalidValue;
        --a.R;
    }
    // A unit's W R n head rows of a tensor are shared out in steps of one row per lane group
    // over the tensor's consumer warps, so a unit takes as long as its busiest warp. Where the
    // block above leaves the warps unevenly loaded, take a larger one (up to twice as many rows,
    // still fitting) that evens them out: e.g. 40 heads of 64 at W = 8, 160 rows per box, give 2
    // or 3 steps per warp; 6 rows give 240, 4 steps for every warp.
    {
        const bool compiled = (p.d & (p.d - 1)) == 0;
        const int P = compiled ? (p.d >= 16 ? 8 : 4) : (p.d % 16 == 0 ? 8 : 4);
        const int g = int(p.d / (2 * P));
        const int per_step = (32 / (compiled ? g : row_lane_stride(g))) * ULY_FT_ILP;
        const int64_t half_nw = kFtConsumerWarps / 2;
        auto balance = [&](int64_t R) {
            const int64_t rows_ = W * R * p.n[0];
            const int64_t steps = (rows_ + per_step - 1) / per_step;
            const int64_t busiest = (steps + half_nw - 1) / half_nw;
            return double(rows_) / double(half_nw * busiest * per_step);
        };
        int64_t best = a.R;
        double best_b = balance(a.R);
        for (int64_t R = a.R + 1; R <= 2 * a.R && R <= 128 && fits(R); ++R) {
            if (balance(R) > best_b + 0.05) {
                best = R;
                best_b = balance(R);
            }
        }
        a.R = best;
    }
    a.box_bytes = uint32_t(a.R * row);
    a.box_stride = uint32_t(up(a.box_bytes, 128));
    a.stage_bytes = 2 * a.box_stride;
    a.table_bytes = uint32_t(up(a.R * (p.d / 2) * 8, 128));
    const int smem = ft_smem_layout(int(p.d), a.table_bytes, a.stage_bytes).total;
    a.W = W;
    a.n = int32_t(p.n[0]);
    a.d = int32_t(p.d);
    a.run = uint32_t(run);
    a.S = p.S;
    a.rms_w = f.rms_w;
    a.eps = f.eps;
    std::memcpy(a.turn_hi, f.turn_hi, sizeof a.turn_hi);
    std::memcpy(a.turn_lo, f.turn_lo, sizeof a.turn_lo);
    int64_t total = 0, total2 = 0;
    for (int k = 0; k < kMaxW; ++k) {
        const bool live = k < W;
        a.q_out[k] = live ? f.q_out[k] : nullptr;
        a.k_out[k] = live ? f.k_out[k] : nullptr;
        for (int pp = 0; pp < n_plain; ++pp)
            a.plain_out[pp][k] = live ? f.plane_out[f.plain_plane[pp]][k] : nullptr;
        a.seq_off[k] = live ? p.seq_off[k] : 0;
        a.row_lo[k] = live ? rows.lo[k] : 0;
        a.rows[k] = live ? rows.cnt[k] : 0;
        a.blocks[k] = (a.rows[k] + a.R - 1) / a.R;
        a.blocks2[k] = (a.rows[k] + 2 * a.R - 1) / (2 * a.R);
        a.unit_begin[k] = total;
        a.unit_begin2[k] = total2;
        total += p.b * a.blocks[k];
        total2 += p.b * a.blocks2[k];
    }
    a.unit_begin[kMaxW] = total;
    a.unit_begin2[kMaxW] = total2;
    a.qk_units = total;
    a.plain_units = total2;
    a.n_plain = n_plain;
    a.total_units = total + n_plain * total2;
    if (a.total_units == 0) return cudaSuccess;
    for (int q = 0; q < W; ++q) {
        if (a.rows[q] == 0) continue;
        const int64_t off = a.row_lo[q] * pitch;
        const int64_t bs = p.s[q] * pitch;
        const uint8_t* qb = packed ? f.packed_in[q] + off + f.q_plane * row : f.q_in[q] + off;
        const uint8_t* kb = packed ? f.packed_in[q] + off + f.k_plane * row : f.k_in[q] + off;
        if (!encode_group_map(&a.qmap[q], qb, run, a.rows[q], W, p.b, pitch, bs, a.R) ||
            !encode_group_map(&a.kmap[q], kb, run, a.rows[q], W, p.b, pitch, bs, a.R))
            return cudaErrorInvalidValue;
        for (int pp = 0; pp < n_plain; ++pp) {
            const uint8_t* pb = f.packed_in[q] + off + f.plain_plane[pp] * row;
            if (!encode_group_map(&a.pmap[pp][q], pb, run, a.rows[q], W, p.b, pitch, bs, 2 * a.R))
                return cudaErrorInvalidValue;
        }
    }
    total = a.total_units;
    int64_t grid = int64_t(sm_count) * ULY_FT_CTAS_PER_SM;
    if (max_grid > 0 && grid > max_grid) grid = max_grid;
    if (grid > total) grid = total;
    const bool f16 = f.elem_f16 != 0, half = f.rope_half != 0;
    switch (p.d) {
        case 8: return ft_launch_variant<8>(a, f16, half, smem, stream, device, int(grid));
        case 16: return ft_launch_variant<16>(a, f16, half, smem, stream, device, int(grid));
        case 32: return ft_launch_variant<32>(a, f16, half, smem, stream, device, int(grid));
        case 64: return ft_launch_variant<64>(a, f16, half, smem, stream, device, int(grid));
        case 128: return ft_launch_variant<128>(a, f16, half, smem, stream, device, int(grid));
        case 256: return ft_launch_variant<256>(a, f16, half, smem, stream, device, int(grid));
        default:  // any other multiple of 8 up to 256: a run-time row layout
            if (p.d % 8 != 0 || p.d < 8 || p.d > kMaxFusedD) return cudaErrorInvalidValue;
            switch (rt_layout_for(int(p.d))) {
                case 0: return ft_launch_variant<0>(a, f16, half, smem, stream, device, int(grid));
                case kRtWide:
                    return ft_launch_variant<kRtWide>(a, f16, half, smem, stream, device, int(grid));
                case kRtPow2:
                    return ft_launch_variant<kRtPow2>(a, f16, half, smem, stream, device, int(grid));
                default:
                    return ft_launch_variant<kRtPow2 | kRtWide>(a, f16, half, smem, stream, device,
                                                                int(grid));
            }
    }
}

cudaError_t fused_tensor_status(unsigned* status, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(status, g_fused_tensor_status, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_fused_tensor_status, &zero, sizeof(unsigned));
}

}  // namespace uly
