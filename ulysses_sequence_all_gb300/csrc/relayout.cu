// relayout.cu -- the Ulysses 4D sequence/head relayout kernels (modes 0 and 1).
//
// The relayout is a permutation of contiguous runs: for every segment (q, r) -- rank q's sequence
// shard and rank r's head group -- and every batch index, row i of rank q's (b, s_q, N, d) tensor
// holds at byte offset head_off(r) * d * e one run of n_r * d * e bytes, and that run is row
// seq_off(q) + i of rank r's (b, S, n_r, d) tensor. On the head side consecutive rows of a
// segment are adjacent, so a block of rows is one contiguous span there and a strided gather on
// the sequence side (fast-ulysses 0.1.0, opening paragraph: the relayout is expressed as copy
// strides instead of separate permute kernels).
//
// Two engines move the same work units:
//  * TMA: a persistent grid, one warp per CTA, a ring of shared-memory stages. Each unit's rows
//    come in through cp.async.bulk (one per strided run, or one for the contiguous span) that
//    complete on the stage's mbarrier, and leave through cp.async.bulk stores. No thread touches
//    the bytes; the SM only issues copies.
//  * VEC: a grid-stride loop of warps, 16-byte vector loads (L1 no-allocate) and stores, several
//    in flight per lane.
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "../../include/ulysses.h"
#include "plan.h"
#include "ptx.cuh"
#include "tensor_map.h"

namespace uly {

static __device__ unsigned g_relayout_status;

#ifndef ULY_TMA_UNIT_BYTES
#define ULY_TMA_UNIT_BYTES 24576
#endif
#ifndef ULY_TMA_STAGES
#define ULY_TMA_STAGES 4
#endif
#ifndef ULY_TMA_CTAS_PER_SM
#define ULY_TMA_CTAS_PER_SM 2
#endif
#ifndef ULY_VEC_UNIT_BYTES
#define ULY_VEC_UNIT_BYTES 16384
#endif
#ifndef ULY_VEC_UNROLL
#define ULY_VEC_UNROLL 4
#endif
// Loads in flight ahead of the unit being stored by the segment kernel (relayout_tma_kernel), per
// mode: mode 0 loads strided runs and stores one span, mode 1 the reverse. The row-tile kernel's
// lookahead is chosen per plan instead (relayout_row_ring).
#ifndef ULY_TMA_LOOKAHEAD0
#define ULY_TMA_LOOKAHEAD0 3
#endif
#ifndef ULY_TMA_LOOKAHEAD1
#define ULY_TMA_LOOKAHEAD1 2
#endif
static_assert(ULY_TMA_LOOKAHEAD0 >= 1 && ULY_TMA_LOOKAHEAD0 <= ULY_TMA_STAGES, "lookahead <= stages");
static_assert(ULY_TMA_LOOKAHEAD1 >= 1 && ULY_TMA_LOOKAHEAD1 <= ULY_TMA_STAGES, "lookahead <= stages");
static_assert(ULY_TMA_STAGES <= 16 && kRowStages <= 16, "stage barriers must fit the barrier area");
constexpr int kTmaBarrierBytes = 128;  // the stage barriers sit before the first stage
constexpr int kVecThreads = 256;

// The stage ring of the TMA kernels (one warp per CTA). Unit k of this CTA lives in stage
// k % K. Loads run L units ahead of the unit being stored; a stage is refilled only when the
// bulk stores that last read it (unit k + L - K, K - L groups back) have finished reading shared
// memory. So up to L loads and K - L store groups are in flight, and the loop never waits on the
// stores it has just issued. Every wait is bounded and its outcome is made uniform across the
// warp (a lane that timed out stops them all); on a timeout the status word records it,
// loads still in flight are waited for (bounded again), and the warp returns.
template <int K, int L, class Load, class Store>
__device__ __forceinline__ void run_stage_ring(uint64_t* full, int64_t n, int lane, Load load,
                                               Store store)
{
    int64_t loaded = n < L ? n : L;
    for (int64_t k = 0; k < loaded; ++k) load(k);
    int64_t k = 0;
    bool ok = true;
    for (; k < n; ++k) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[k % K], uint32_t((k / K) & 1)))) {
            ok = false;
            break;
        }
        store(k);
        bulk_commit();
        if (loaded < n) {
            bulk_wait_read<K - L>();
            __syncwarp();
            load(loaded);
            ++loaded;
        }
    }
    if (!ok) {
        if (lane == 0) atomicOr(&g_relayout_status, kStatusWaitTimeout);
        for (int64_t j = k; j < loaded; ++j) {
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[j % K], uint32_t((j / K) & 1)))) {
                if (lane == 0) atomicOr(&g_relayout_status, kStatusDrainTimeout);
                break;
            }
        }
    }
    bulk_wait<0>();
}

struct Unit {
    int q, r;
    int64_t bb, i0, nrows, col0, cols;
};

// Largest segment g with unit_begin[g] <= u; segments without units share a prefix value with
// their successor, so the match always owns unit u.
__device__ __forceinline__ int find_segment(const RelayoutArgs& a, int64_t u)
{
    int lo = 0, hi = a.W * a.W - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.unit_begin[mid] <= u)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ Unit decode(const RelayoutArgs& a, int64_t u)
{
    Unit t;
    const int g = find_segment(a, u);
    t.q = g / a.W;
    t.r = g - t.q * a.W;
    const int64_t local = u - a.unit_begin[g];
    const int64_t R = a.rows_per_unit[t.r];
    const int64_t P = a.pieces[t.r];
    const int64_t rows = a.rows[t.q];
    const int64_t per_batch = ((rows + R - 1) / R) * P;
    t.bb = div_fast(local, per_batch);
    const int64_t rem = local - t.bb * per_batch;
    const int64_t blk = div_fast(rem, P);
    const int64_t piece = rem - blk * P;
    const int64_t i0 = blk * R;
    t.nrows = min(R, rows - i0);
    t.i0 = a.row_lo[t.q] + i0;
    const int64_t run = a.n[t.r] * a.d_bytes;
    t.col0 = piece * a.unit_bytes;
    t.cols = (P == 1) ? run : min(int64_t(a.unit_bytes), run - t.col0);
    return t;
}

// Row k of unit t on rank q's (b, s_q, N, d) tensor.
__device__ __forceinline__ uint8_t* seq_addr(const RelayoutArgs& a, const Unit& t, int64_t k)
{
    return a.seq_ptr[t.q] + ((t.bb * a.s[t.q] + t.i0 + k) * a.N + a.head_off[t.r]) * a.d_bytes + t.col0;
}

// Row k of unit t on rank r's (b, S, n_r, d) tensor (rows are adjacent: pitch n_r * d * e).
__device__ __forceinline__ uint8_t* head_addr(const RelayoutArgs& a, const Unit& t, int64_t k)
{
    return a.head_ptr[t.r] + ((t.bb * a.S + a.seq_off[t.q] + t.i0 + k) * a.n[t.r]) * a.d_bytes +
           t.col0;
}

template <int MODE>
__global__ void __launch_bounds__(32, 1) relayout_tma_kernel(const __grid_constant__ RelayoutArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int K = ULY_TMA_STAGES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint8_t* stage0 = smem + kTmaBarrierBytes;
    const int lane = threadIdx.x;
    const int64_t first = blockIdx.x, step = gridDim.x;
    const int64_t n = first < a.total_units ? (a.total_units - 1 - first) / step + 1 : 0;
    if (n == 0) return;
    if (lane == 0) {
        for (int s = 0; s < K; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    __syncwarp();

    auto issue_load = [&](int64_t k) {
        const Unit t = decode(a, first + k * step);
        const int s = int(k % K);
        uint8_t* dst = stage0 + size_t(s) * ULY_TMA_UNIT_BYTES;
        const uint32_t bytes = uint32_t(t.nrows * t.cols);
        if (lane == 0) mbar_arrive_expect_tx(&full[s], bytes);
        __syncwarp();
        if (MODE == 0) {  // strided runs of the sequence side, packed back to back
            for (int64_t row = lane; row < t.nrows; row += 32)
                bulk_g2s(dst + row * t.cols, seq_addr(a, t, row), uint32_t(t.cols), &full[s]);
        } else {  // one contiguous span of the head side
            if (lane == 0) bulk_g2s(dst, head_addr(a, t, 0), bytes, &full[s]);
        }
    };
    auto issue_store = [&](int64_t k) {
        const Unit t = decode(a, first + k * step);
        const uint8_t* src = stage0 + size_t(k % K) * ULY_TMA_UNIT_BYTES;
        if (MODE == 0) {
            if (lane == 0) bulk_s2g(head_addr(a, t, 0), src, uint32_t(t.nrows * t.cols));
        } else {
            for (int64_t row = lane; row < t.nrows; row += 32)
                bulk_s2g(seq_addr(a, t, row), src + row * t.cols, uint32_t(t.cols));
        }
    };
    run_stage_ring<ULY_TMA_STAGES, MODE == 0 ? ULY_TMA_LOOKAHEAD0 : ULY_TMA_LOOKAHEAD1>(
        full, n, lane, issue_load, issue_store);
}

// ---- tensor engine: one tensor-map box per unit on the strided side --------------------------------
// A unit is a block of up to R consecutive rows of one sequence shard q and batch index, for one
// head group r: on the sequence side R runs of n_r d e bytes, strided by N d e; on the head side one
// contiguous span. The strided side moves with one tiled tensor copy instead of one bulk copy per
// row: for segment g = (q, r) a 3-D tensor map describes rank q's runs of head group r in this
// launch's rows, (run / 8 eight-byte elements, chunk rows, b) with strides (N d e, s_q N d e) bytes,
// starting at the run's first byte, so every box starts at x = 0. Mode 0: one tensor load of the
// unit's rows (rows past the chunk are filled, not read from elsewhere) and one bulk store of the
// contiguous head-side span; mode 1: one bulk load of the span and one tensor store, which the map
// clips at the chunk's rows. Units are ordered (shard, batch index, row block, head group), so
// consecutive units cover the same rows and the grid as a whole reads and writes whole rows in
// sequence. R (at most 256, the box limit) is the same for every head group: the rows of the
// widest run that fit a stage; a run is at most 2,048 bytes (256 eight-byte elements), and plans
// with longer runs use the other engines.
//
// A unit costs a CTA about half a microsecond whatever its size (16 to 52 KiB measured), so a
// CTA's throughput grows with its stage bytes, while a full grid of small stages spreads the
// traffic more evenly. Two pipeline shapes per mode, one CTA per SM (stages fill shared memory):
// a full grid takes many 24 KiB stages with most of them loading; a grid capped below the SM
// count (the relayout sharing the GPU with other work) takes four stages of about 50 KiB, which
// keeps 6 TB/s on half the SMs at the Wan-720p shape.
struct TensorArgs {
    CUtensorMap map[kMaxSeg];  // segment g = q * W + r
    uint8_t* seq_ptr[kMaxW];
    uint8_t* head_ptr[kMaxW];
    int64_t s[kMaxW], seq_off[kMaxW], n[kMaxW], head_off[kMaxW];
    int64_t row_lo[kMaxW], rows[kMaxW];  // this launch's rows of shard q
    int64_t blocks[kMaxW];               // row blocks per batch index of shard q
    int64_t unit_begin[kMaxW + 1];       // prefix of unit counts over q
    int64_t S, N, b, d_bytes, R, total_units;
    int32_t live_r[kMaxW];  // head groups with n_r > 0, in order
    int32_t W, n_live;
};

struct TensorUnit {
    int q, r;
    int64_t bb, i0, nrows, run;
};

__device__ __forceinline__ TensorUnit decode_tensor(const TensorArgs& a, int64_t u)
{
    int lo = 0, hi = a.W - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.unit_begin[mid] <= u)
            lo = mid;
        else
            hi = mid - 1;
    }
    TensorUnit t;
    t.q = lo;
    const int64_t local = u - a.unit_begin[lo];
    const int64_t rest = div_fast(local, a.n_live);
    t.r = a.live_r[local - rest * a.n_live];
    const int64_t blocks = a.blocks[lo];
    t.bb = div_fast(rest, blocks);
    const int64_t blk = rest - t.bb * blocks;
    t.i0 = blk * a.R;  // in the chunk
    t.nrows = min(a.R, a.rows[lo] - t.i0);
    t.run = a.n[t.r] * a.d_bytes;
    return t;
}

constexpr int kTensorStageAlign = 1024;  // stage buffers start here (tensor copies want 128 B)

struct TensorShape {
    int stages, unit_bytes, lookahead;
};
// [mode]: measured at the Wan-720p shape (W = 8, runs of 1,280 bytes), CUDA events back to back.
constexpr TensorShape kTensorFull[2] = {{8, 24576, 7}, {9, 24576, 4}};
constexpr TensorShape kTensorCapped[2] = {{4, 53248, 3}, {4, 49152, 3}};

constexpr int tensor_smem(TensorShape t) { return kTensorStageAlign + t.stages * t.unit_bytes; }

template <int MODE, int K, int UNIT, int L>
__global__ void __launch_bounds__(32, 1) relayout_tensor_kernel(const __grid_constant__ TensorArgs a)
{
    static_assert(UNIT % 1024 == 0, "tensor-copy stages must stay 1024-byte aligned");
    static_assert(L >= 1 && L <= K && K <= 16, "lookahead <= stages; barriers fit the area");
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint8_t* stage0 = smem + kTensorStageAlign;
    const int lane = threadIdx.x;
    const int64_t first = blockIdx.x, step = gridDim.x;
    const int64_t n = first < a.total_units ? (a.total_units - 1 - first) / step + 1 : 0;
    if (n == 0) return;
    if (lane == 0) {
        for (int s = 0; s < K; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    __syncwarp();
    // the unit's contiguous span on rank r's (b, S, n_r, d) head side
    auto head_span = [&](const TensorUnit& t) {
        return a.head_ptr[t.r] +
               (t.bb * a.S + a.seq_off[t.q] + a.row_lo[t.q] + t.i0) * t.run;
    };
    auto issue_load = [&](int64_t k) {
        if (lane != 0) return;
        const TensorUnit t = decode_tensor(a, first + k * step);
        const int s = int(k % K);
        uint8_t* dst = stage0 + size_t(s) * UNIT;
        if (MODE == 0) {  // the whole box arrives (rows past the chunk are filled)
            mbar_arrive_expect_tx(&full[s], uint32_t(a.R * t.run));
            tensor_g2s_3d(dst, &a.map[t.q * a.W + t.r], 0, int(t.i0), int(t.bb), &full[s]);
        } else {
            const uint32_t bytes = uint32_t(t.nrows * t.run);
            mbar_arrive_expect_tx(&full[s], bytes);
            bulk_g2s(dst, head_span(t), bytes, &full[s]);
        }
    };
    auto issue_store = [&](int64_t k) {
        if (lane != 0) return;
        const TensorUnit t = decode_tensor(a, first + k * step);
        const uint8_t* src = stage0 + size_t(k % K) * UNIT;
        if (MODE == 0)
            bulk_s2g(head_span(t), src, uint32_t(t.nrows * t.run));
        else
            tensor_s2g_3d(&a.map[t.q * a.W + t.r], 0, int(t.i0), int(t.bb), src);
    };
    run_stage_ring<K, L>(full, n, lane, issue_load, issue_store);
}

// ---- row tiles: whole rows through shared memory ------------------------------------------------
// Unit = up to tile_rows consecutive rows of shard q, batch bb. Shared memory holds the rows in
// their sequence-side layout (row i, all N heads). Mode 0: one bulk load of the contiguous
// sequence-side span, then one bulk store per (row, destination rank) run; the runs of one rank
// are adjacent in its tensor, so each rank receives one contiguous span per unit. Mode 1 mirrors
// this: one bulk load per (row, source rank) run, one bulk store of the contiguous span. Both
// sides are therefore streamed in long sequential spans across the grid.
struct RowTile {
    int q;
    int64_t bb, i0, nrows;
};

__device__ __forceinline__ RowTile decode_rows(const RowTileArgs& a, int64_t u)
{
    int lo = 0, hi = a.W - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.unit_begin[mid] <= u)
            lo = mid;
        else
            hi = mid - 1;
    }
    RowTile t;
    t.q = lo;
    const int64_t T = a.tile_rows;
    const int64_t rows = a.rows[lo];
    const int64_t blocks = (rows + T - 1) / T;
    const int64_t local = u - a.unit_begin[lo];
    t.bb = div_fast(local, blocks);
    const int64_t blk = local - t.bb * blocks;
    t.i0 = a.row_lo[lo] + blk * T;
    t.nrows = min(T, rows - blk * T);
    return t;
}

template <int MODE, int L>
__global__ void __launch_bounds__(32, 1) relayout_rows_kernel(const __grid_constant__ RowTileArgs a)
{
    static_assert(L >= 1 && L <= kRowStages, "lookahead <= stages");
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int K = kRowStages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint8_t* stage0 = smem + kTmaBarrierBytes;
    const int lane = threadIdx.x;
    const int64_t first = blockIdx.x, step = gridDim.x;
    const int64_t n = first < a.total_units ? (a.total_units - 1 - first) / step + 1 : 0;
    if (n == 0) return;
    if (lane == 0) {
        for (int s = 0; s < K; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    __syncwarp();
    const int W = a.W;
    const int64_t row_bytes = a.N * a.d_bytes;

    // sequence side: nrows whole rows, contiguous
    auto seq_span = [&](const RowTile& t) {
        return a.seq_ptr[t.q] + (t.bb * a.s[t.q] + t.i0) * row_bytes;
    };
    // head side of rank r: nrows runs of n_r * d * e bytes, contiguous
    auto head_span = [&](const RowTile& t, int r) {
        return a.head_ptr[r] + (t.bb * a.S + a.seq_off[t.q] + t.i0) * a.n[r] * a.d_bytes;
    };

    auto issue_load = [&](int64_t k) {
        const RowTile t = decode_rows(a, first + k * step);
        const int s = int(k % K);
        uint8_t* stage = stage0 + size_t(s) * a.stage_bytes;
        const uint32_t bytes = uint32_t(t.nrows * row_bytes);
        if (lane == 0) mbar_arrive_expect_tx(&full[s], bytes);
        __syncwarp();
        if (MODE == 0) {
            if (lane == 0) bulk_g2s(stage, seq_span(t), bytes, &full[s]);
        } else {
            const int pairs = int(t.nrows) * W;
            for (int idx = lane; idx < pairs; idx += 32) {
                const int i = idx / W, r = idx - (idx / W) * W;
                const int64_t run = a.n[r] * a.d_bytes;
                if (run == 0) continue;
                bulk_g2s(stage + i * row_bytes + a.head_off[r] * a.d_bytes, head_span(t, r) + i * run,
                         uint32_t(run), &full[s]);
            }
        }
    };
    auto issue_store = [&](int64_t k) {
        const RowTile t = decode_rows(a, first + k * step);
        const uint8_t* stage = stage0 + size_t(k % K) * a.stage_bytes;
        if (MODE == 0) {
            const int pairs = int(t.nrows) * W;
            for (int idx = lane; idx < pairs; idx += 32) {
                const int i = idx / W, r = idx - (idx / W) * W;
                const int64_t run = a.n[r] * a.d_bytes;
                if (run == 0) continue;
                bulk_s2g(head_span(t, r) + i * run, stage + i * row_bytes + a.head_off[r] * a.d_bytes,
                         uint32_t(run));
            }
        } else {
            if (lane == 0) bulk_s2g(seq_span(t), stage, uint32_t(t.nrows * row_bytes));
        }
    };
    run_stage_ring<K, L>(full, n, lane, issue_load, issue_store);
}

template <int MODE>
__global__ void __launch_bounds__(kVecThreads) relayout_vec_kernel(const __grid_constant__ RelayoutArgs a)
{
    constexpr int U = ULY_VEC_UNROLL;
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    for (int64_t u = warp; u < a.total_units; u += nwarps) {
        const Unit t = decode(a, u);
        const uint8_t* seq0 = seq_addr(a, t, 0);
        const uint8_t* head0 = head_addr(a, t, 0);
        const int64_t seq_pitch = a.N * a.d_bytes;
        const int64_t head_pitch = a.n[t.r] * a.d_bytes;
        const uint8_t* src = MODE == 0 ? seq0 : head0;
        uint8_t* dst = const_cast<uint8_t*>(MODE == 0 ? head0 : seq0);
        const int64_t src_pitch = MODE == 0 ? seq_pitch : head_pitch;
        const int64_t dst_pitch = MODE == 0 ? head_pitch : seq_pitch;
        const uint32_t vpr = uint32_t(t.cols >> 4);  // 16-byte vectors per row
        const uint32_t total = uint32_t(t.nrows) * vpr;
        // lane's (row, vector) and its advance per 32 vectors, kept without per-step division
        uint32_t k = lane / vpr, c = lane % vpr;
        const uint32_t dk = 32 / vpr, dc = 32 % vpr;
        for (uint32_t v0 = 0; v0 < total; v0 += 32 * U) {
            uint4 buf[U];
            uint32_t kk[U], cc[U];
#pragma unroll
            for (int j = 0; j < U; ++j) {
                kk[j] = k;
                cc[j] = c;
                if (v0 + j * 32 + lane < total) buf[j] = ld_stream_v4(src + k * src_pitch + c * 16);
                k += dk;
                c += dc;
                if (c >= vpr) {
                    c -= vpr;
                    k += 1;
                }
            }
#pragma unroll
            for (int j = 0; j < U; ++j)
                if (v0 + j * 32 + lane < total) st_v4(dst + kk[j] * dst_pitch + cc[j] * 16, buf[j]);
        }
    }
}

int64_t relayout_unit_bytes(int engine) { return engine == ULY_ENGINE_VEC ? ULY_VEC_UNIT_BYTES : ULY_TMA_UNIT_BYTES; }

// per device: whether the TMA kernels' shared-memory limit has been raised (any host thread)
static std::atomic<int> g_smem_set[64];

// Raise every TMA kernel's dynamic shared-memory limit to the per-CTA maximum, once per device.
static cudaError_t ensure_tma_smem(int device)
{
    if (device < 0 || device >= 64 || g_smem_set[device].load()) return cudaSuccess;
    const void* kernels[] = {reinterpret_cast<const void*>(relayout_tma_kernel<0>),
                             reinterpret_cast<const void*>(relayout_tma_kernel<1>),
                             reinterpret_cast<const void*>(relayout_rows_kernel<0, 2>),
                             reinterpret_cast<const void*>(relayout_rows_kernel<0, 3>),
                             reinterpret_cast<const void*>(relayout_rows_kernel<1, 2>),
                             reinterpret_cast<const void*>(relayout_rows_kernel<1, 3>)};
    for (const void* k : kernels) {
        cudaError_t e =
            cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemPerCtaMax);
        if (e != cudaSuccess) return e;
    }
    g_smem_set[device].store(1);
    return cudaSuccess;
}

constexpr int kTmaSmem = kTmaBarrierBytes + ULY_TMA_STAGES * ULY_TMA_UNIT_BYTES;
static_assert(kTmaSmem <= kSmemPerCtaMax, "segment ring must fit one CTA");

cudaError_t relayout_launch(const RelayoutArgs& a, int mode, int engine, cudaStream_t stream,
                            int device, int sm_count, int64_t max_grid)
{
    if (a.total_units == 0) return cudaSuccess;
    if (engine == ULY_ENGINE_VEC) {
        static std::atomic<int> vec_blocks_per_sm{0};  // the same on every GB300; any thread
        int blocks_per_sm = vec_blocks_per_sm.load();
        if (blocks_per_sm == 0) {
            int nb = 0;
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, relayout_vec_kernel<0>, kVecThreads, 0);
            blocks_per_sm = nb > 0 ? nb : 1;
            vec_blocks_per_sm.store(blocks_per_sm);
        }
        const int64_t warps_needed = a.total_units;
        int64_t grid = int64_t(sm_count) * blocks_per_sm;
        if (max_grid > 0 && grid > max_grid) grid = max_grid;
        const int64_t useful = (warps_needed * 32 + kVecThreads - 1) / kVecThreads;
        if (grid > useful) grid = useful;
        if (mode == 0)
            relayout_vec_kernel<0><<<unsigned(grid), kVecThreads, 0, stream>>>(a);
        else
            relayout_vec_kernel<1><<<unsigned(grid), kVecThreads, 0, stream>>>(a);
        return cudaGetLastError();
    }
    cudaError_t e = ensure_tma_smem(device);
    if (e != cudaSuccess) return e;
    int64_t grid = int64_t(sm_count) * ULY_TMA_CTAS_PER_SM;
    if (max_grid > 0 && grid > max_grid) grid = max_grid;
    if (grid > a.total_units) grid = a.total_units;
    if (mode == 0)
        relayout_tma_kernel<0><<<unsigned(grid), 32, kTmaSmem, stream>>>(a);
    else
        relayout_tma_kernel<1><<<unsigned(grid), 32, kTmaSmem, stream>>>(a);
    return cudaGetLastError();
}

// The tensor-map encoder of the driver, fetched once through the runtime (no link to libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool encode_run_map(CUtensorMap* map, const void* base, int64_t run, int64_t rows, int64_t b,
                    int64_t row_stride, int64_t batch_stride, int64_t box_rows)
{
    EncodeTiledFn encode = encode_tiled_fn();
    if (!encode) return false;
    const cuuint64_t dims[3] = {cuuint64_t(run / 8), cuuint64_t(rows), cuuint64_t(b)};
    const cuuint64_t strides[2] = {cuuint64_t(row_stride), cuuint64_t(batch_stride)};
    const cuuint32_t boxdim[3] = {cuuint32_t(run / 8), cuuint32_t(box_rows), 1};
    const cuuint32_t estrides[3] = {1, 1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<void*>(base), dims, strides,
                  boxdim, estrides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_group_map(CUtensorMap* map, const void* base, int64_t run, int64_t rows, int64_t W,
                      int64_t b, int64_t row_stride, int64_t batch_stride, int64_t box_rows)
{
    EncodeTiledFn encode = encode_tiled_fn();
    if (!encode) return false;
    const cuuint64_t dims[4] = {cuuint64_t(run / 8), cuuint64_t(rows), cuuint64_t(W), cuuint64_t(b)};
    const cuuint64_t strides[3] = {cuuint64_t(row_stride), cuuint64_t(run), cuuint64_t(batch_stride)};
    const cuuint32_t boxdim[4] = {cuuint32_t(run / 8), cuuint32_t(box_rows), cuuint32_t(W), 1};
    const cuuint32_t estrides[4] = {1, 1, 1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 4, const_cast<void*>(base), dims, strides,
                  boxdim, estrides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, int K, int UNIT, int L>
static cudaError_t tensor_launch_shape(const TensorArgs& a, unsigned grid, cudaStream_t stream,
                                       int device)
{
    auto kernel = relayout_tensor_kernel<MODE, K, UNIT, L>;
    constexpr int smem = tensor_smem({K, UNIT, L});
    static std::atomic<int> smem_set[64];
    if (device >= 0 && device < 64 && !smem_set[device].load()) {
        const cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        smem_set[device].store(1);
    }
    kernel<<<grid, 32, smem, stream>>>(a);
    return cudaGetLastError();
}

#define ULY_TENSOR_SHAPE(M, T) M, T.stages, T.unit_bytes, T.lookahead

static cudaError_t tensor_dispatch(int mode, bool capped, const TensorArgs& a, unsigned grid,
                                   cudaStream_t stream, int device)
{
    if (mode == 0)
        return capped ? tensor_launch_shape<ULY_TENSOR_SHAPE(0, kTensorCapped[0])>(a, grid, stream, device)
                      : tensor_launch_shape<ULY_TENSOR_SHAPE(0, kTensorFull[0])>(a, grid, stream, device);
    return capped ? tensor_launch_shape<ULY_TENSOR_SHAPE(1, kTensorCapped[1])>(a, grid, stream, device)
                  : tensor_launch_shape<ULY_TENSOR_SHAPE(1, kTensorFull[1])>(a, grid, stream, device);
}
#undef ULY_TENSOR_SHAPE

// Whether the tensor engine takes this plan: every run of at most 256 eight-byte elements.
bool relayout_tensor_fits(const Plan& p)
{
    for (int r = 0; r < p.W; ++r)
        if (p.n[r] * p.d * p.e > 256 * 8) return false;
    return true;
}

// The automatic engine's choice. A tensor unit costs a CTA a fixed time, so the engine wins where
// its units fill their stages: every head group's run equally long (measured: 1.03x the row tiles
// at the Wan-720p shape; 0.85-0.99x on plans with unequal head splits, whose smaller groups leave
// stages part-empty). Under a CTA cap below the SM count it wins on every plan it takes (measured
// 2.3 to 5.3 times the row tiles' throughput at caps of 114, 76 and 38 CTAs), as its CTAs keep
// more bytes in flight.
bool relayout_tensor_preferred(const Plan& p, int sm_count)
{
    if (!relayout_tensor_fits(p)) return false;
    if (p.max_ctas > 0 && p.max_ctas < sm_count) return true;
    int64_t run = 0;
    for (int r = 0; r < p.W; ++r) {
        if (p.n[r] == 0) continue;
        if (run != 0 && p.n[r] != run) return false;
        run = p.n[r];
    }
    return true;
}

cudaError_t relayout_tensor_launch(const Plan& p, const ChunkRows& rows, uint8_t* const* seq,
                                   uint8_t* const* head, int mode, cudaStream_t stream, int device,
                                   int sm_count, int64_t max_grid)
{
    TensorArgs a;
    std::memset(&a, 0, sizeof a);
    const int W = p.W;
    const int64_t de = p.d * p.e;
    int64_t max_run = 0;
    a.n_live = 0;
    for (int r = 0; r < W; ++r) {
        if (p.n[r] == 0) continue;
        a.live_r[a.n_live++] = r;
        if (p.n[r] * de > max_run) max_run = p.n[r] * de;
    }
    if (a.n_live == 0) return cudaSuccess;
    // one CTA per SM; a cap below the SM count takes the large-stage shape
    int64_t grid = sm_count;
    if (max_grid > 0 && grid > max_grid) grid = max_grid;
    const bool capped = grid < sm_count;
    const TensorShape shape = capped ? kTensorCapped[mode] : kTensorFull[mode];
    a.R = shape.unit_bytes / max_run;
    if (a.R > 256) a.R = 256;
    a.W = W;
    a.S = p.S;
    a.N = p.N;
    a.b = p.b;
    a.d_bytes = de;
    int64_t total = 0;
    for (int k = 0; k < kMaxW; ++k) {
        const bool live = k < W;
        a.seq_ptr[k] = live ? seq[k] : nullptr;
        a.head_ptr[k] = live ? head[k] : nullptr;
        a.s[k] = live ? p.s[k] : 0;
        a.seq_off[k] = live ? p.seq_off[k] : 0;
        a.n[k] = live ? p.n[k] : 0;
        a.head_off[k] = live ? p.head_off[k] : 0;
        a.row_lo[k] = live ? rows.lo[k] : 0;
        a.rows[k] = live ? rows.cnt[k] : 0;
        a.blocks[k] = (a.rows[k] + a.R - 1) / a.R;
        a.unit_begin[k] = total;
        total += p.b * a.blocks[k] * a.n_live;
    }
    a.unit_begin[kMaxW] = total;
    a.total_units = total;
    if (total == 0) return cudaSuccess;
    for (int q = 0; q < W; ++q) {
        for (int r = 0; r < W; ++r) {
            const int64_t run = a.n[r] * de;
            if (a.rows[q] == 0 || run == 0) continue;
            const uint8_t* base = a.seq_ptr[q] + (a.row_lo[q] * a.N + a.head_off[r]) * de;
            if (!encode_run_map(&a.map[q * W + r], base, run, a.rows[q], a.b, a.N * de,
                                a.s[q] * a.N * de, a.R))
                return cudaErrorInvalidValue;
        }
    }
    if (grid > a.total_units) grid = a.total_units;
    return tensor_dispatch(mode, capped, a, unsigned(grid), stream, device);
}

// The row-tile kernel's pipeline shape for a plan and mode, from its geometry: `row` = one
// token's bytes (N d e), `run` = the mean bytes of one (token, rank) run (row / W), `unit` = the
// whole rows that fit a 24 KiB stage. Measured on a GB300 (CUDA events, the uneven configurations
// of fp8 / fp16 / fp32 at W = 3, 5, 7, 8, the Wan shape and the long packed-QKV shape):
//  * runs below ~900 bytes (fp8 at W >= 6): bulk copies are small and many, and three CTAs per SM
//    with 18 KiB stages, two loads ahead in both modes, beat the default by 12-25%;
//  * units below 20 KiB (one row of 12-20 KiB, as at 56 heads of bf16): three loads ahead in both
//    modes (mode 1 of the long packed-QKV shape +12%);
//  * otherwise mode 0 keeps three loads ahead while the runs are short (1,280 bytes at the Wan
//    shape) and two from ~1,400 bytes on, where its long stores take longer to leave shared
//    memory and want more of the ring (+11-16% at W = 3, 5 and for fp32); mode 1 keeps two.
RowRing relayout_row_ring(const Plan& p, int mode)
{
    const int64_t row = p.N * p.d * p.e;
    const int64_t run = row / p.W;
    RowRing r;
    r.ctas_per_sm = 2;
    r.stage_bytes = 24576;
    if (run < 900) {
        r.ctas_per_sm = 3;
        r.stage_bytes = 18432;
        r.lookahead = 2;
        return r;
    }
    const int64_t unit = row <= r.stage_bytes ? (r.stage_bytes / row) * row : 0;
    if (unit > 0 && unit < 20480)
        r.lookahead = 3;
    else
        r.lookahead = mode == 0 && run < 1400 ? 3 : 2;
    return r;
}

// Rows per tile for the row-tile kernel, 0 when one row does not fit a stage.
int64_t relayout_tile_rows(int64_t row_bytes, int64_t stage_bytes)
{
    return row_bytes <= stage_bytes ? stage_bytes / row_bytes : 0;
}

cudaError_t relayout_rows_launch(const RowTileArgs& a, int mode, const RowRing& ring,
                                 cudaStream_t stream, int device, int sm_count, int64_t max_grid)
{
    if (a.total_units == 0) return cudaSuccess;
    const int smem = kTmaBarrierBytes + kRowStages * ring.stage_bytes;
    if (smem > kSmemPerCtaMax ||
        ring.ctas_per_sm * (smem + kSmemReservedPerCta) > kSmemPerSm ||
        (ring.lookahead != 2 && ring.lookahead != 3) || a.stage_bytes != ring.stage_bytes)
        return cudaErrorInvalidValue;
    cudaError_t e = ensure_tma_smem(device);
    if (e != cudaSuccess) return e;
    int64_t grid = int64_t(sm_count) * ring.ctas_per_sm;
    if (max_grid > 0 && grid > max_grid) grid = max_grid;
    if (grid > a.total_units) grid = a.total_units;
    const unsigned g = unsigned(grid);
    if (mode == 0) {
        if (ring.lookahead == 3)
            relayout_rows_kernel<0, 3><<<g, 32, smem, stream>>>(a);
        else
            relayout_rows_kernel<0, 2><<<g, 32, smem, stream>>>(a);
    } else {
        if (ring.lookahead == 3)
            relayout_rows_kernel<1, 3><<<g, 32, smem, stream>>>(a);
        else
            relayout_rows_kernel<1, 2><<<g, 32, smem, stream>>>(a);
    }
    return cudaGetLastError();
}

// Failure-path self-test: one warp waits on a barrier nothing ever arrives on, gives up after
// limit_ns, records the timeout in the status word and returns like any kernel that timed out.
__global__ void __launch_bounds__(32, 1) selftest_timeout_kernel(uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t never;
    if (threadIdx.x == 0) {
        mbar_init(&never, 1);
        fence_barrier_init();
    }
    __syncwarp();
    if (!mbar_wait_bounded(&never, 0u, limit_ns) && threadIdx.x == 0)
        atomicOr(&g_relayout_status, kStatusWaitTimeout);
}

cudaError_t selftest_timeout_launch(uint64_t limit_ns, cudaStream_t stream)
{
    selftest_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

cudaError_t relayout_status(unsigned* status, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(status, g_relayout_status, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_relayout_status, &zero, sizeof(unsigned));
}

}  // namespace uly
