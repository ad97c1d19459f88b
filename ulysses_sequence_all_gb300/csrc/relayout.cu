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

#include "../../include/ulysses.h"
#include "plan.h"
#include "ptx.cuh"

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
