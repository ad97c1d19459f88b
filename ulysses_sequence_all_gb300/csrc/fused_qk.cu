// fused_qk.cu -- mode-0 relayout of q and k with QK RMSNorm + RoPE applied in the scatter
// (fast-ulysses 0.1.0, "Fusion examples": QK RMSNorm + RoPE inside the scatter kernel).
//
// Per head row x of d bf16 values at global sequence position p:
//     y = x / sqrt(mean(x^2) + eps) * w,   (y[2j], y[2j+1]) rotated by p * theta^(-2j/d),
// in fp32, rounded once to bf16 (nearest even), and written where mode 0 places the row.
//
// Structure: a persistent grid with one CTA per SM and a ring of shared-memory stages.
//  * Warp 0 produces. Per work unit (a few consecutive tokens of one source rank: all N heads of
//    q and of k, two contiguous spans) its lanes first fill the stage's cos/sin table for those
//    tokens' positions, then lane 0 starts the two cp.async.bulk loads. All 32 lanes arrive on
//    the stage's "full" mbarrier (lane 0 with the expected transaction bytes), so a consumer that
//    sees the phase complete sees both the table and the data.
//  * The consumer warps split a stage's head rows into contiguous ranges. A group of d/8 lanes
//    holds one head row (8 values per lane) and each group keeps two rows in flight; the sum of
//    squares is reduced with xor shuffles inside the group, the weight and rotation are applied in
//    registers, and each lane stores 16 bytes straight to the destination rank (a head row is one
//    contiguous 2d-byte span there). Each consumer warp then arrives on the stage's "empty"
//    mbarrier so the producer can refill it.
//
// RoPE angles: p * theta^(-2j/d) reaches ~75,600 rad at the Wan shape, where an fp32 product
// alone is off by ~5e-3 rad. The angle is formed in turns (units of 2 pi): the host supplies
// theta^(-2j/d) / (2 pi) as a float pair hi + lo; p * hi is split exactly into a product and its
// fma residual (Dekker's error-free product via fma), the whole turns are dropped (exact), the
// small terms are added, and sincospif is called on the reduced fraction. The angle error stays
// near 1e-6 rad.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/ulysses.h"
#include "plan.h"
#include "ptx.cuh"

namespace uly {

static __device__ unsigned g_fused_status;

#ifndef ULY_FUSED_CONSUMER_WARPS
#define ULY_FUSED_CONSUMER_WARPS 16
#endif
#ifndef ULY_FUSED_STAGE_TARGET
#define ULY_FUSED_STAGE_TARGET 40960
#endif
#ifndef ULY_FUSED_MAX_STAGES
#define ULY_FUSED_MAX_STAGES 4
#endif
constexpr int kFusedMaxStages = ULY_FUSED_MAX_STAGES;
constexpr int kFusedSmemBudget = 210 * 1024;
constexpr int kFusedHeader = 128;  // 2 * kFusedMaxStages barriers
constexpr int kFusedThreads = 32 * (1 + ULY_FUSED_CONSUMER_WARPS);
constexpr int kFusedMaxHeads = 1024;
constexpr int kIlp = 2;  // head rows in flight per lane group

struct FusedUnit {
    int q;
    int64_t bb, i0;
    int ntok;
};

__device__ __forceinline__ FusedUnit fused_decode(const FusedArgs& a, int64_t u)
{
    int lo = 0, hi = a.W - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.unit_begin[mid] <= u)
            lo = mid;
        else
            hi = mid - 1;
    }
    FusedUnit t;
    t.q = lo;
    const int64_t T = a.tokens_per_unit;
    const int64_t rows = a.rows[lo];
    const int64_t blocks = (rows + T - 1) / T;
    const int64_t local = u - a.unit_begin[lo];
    t.bb = local / blocks;
    const int64_t blk = local - t.bb * blocks;
    t.i0 = a.row_lo[lo] + blk * T;
    t.ntok = int(min(T, rows - blk * T));
    return t;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// cos and sin of 2 pi * frac(p * (hi + lo)), p a non-negative integer below 2^24.
__device__ __forceinline__ float2 rope_cos_sin(float p, float hi, float lo)
{
    const float ph = p * hi;
    const float pe = fmaf(p, hi, -ph);  // exact residual of the product
    float f = ph - rintf(ph);           // exact: drops whole turns
    f += fmaf(p, lo, pe);
    float s, c;
    sincospif(2.0f * f, &s, &c);
    return make_float2(c, s);
}

// Shared-memory layout (byte offsets), shared by the kernel and its launcher.
struct FusedSmem {
    int turns;      // float2 (hi, lo) per pair j < d/2
    int heads;      // int per global head: destination rank << 16 | local head index
    int tables;     // per stage: float2 (cos, sin) per (token, pair)
    int stages;     // per stage: q span then k span
    int table_bytes;
    int total;
};

__host__ __device__ inline FusedSmem fused_smem_layout(int d, int64_t N, int tokens, int stages,
                                                       uint32_t stage_bytes)
{
    auto up = [](int x) { return (x + 127) & ~127; };
    FusedSmem m;
    m.turns = kFusedHeader;
    m.heads = up(m.turns + (d / 2) * 8);
    m.tables = up(m.heads + int(N) * 4);
    m.table_bytes = up(tokens * (d / 2) * 8);
    m.stages = up(m.tables + stages * m.table_bytes);
    m.total = m.stages + stages * int(stage_bytes);
    return m;
}

template <int G>  // lanes per head row; d = 8 * G
__global__ void __launch_bounds__(kFusedThreads, 1) fused_qk_kernel(const __grid_constant__ FusedArgs a)
{
    constexpr int D = 8 * G;
    constexpr int HALF = D / 2;
    constexpr int GPW = 32 / G;         // head rows per warp per slot
    constexpr int PER_STEP = GPW * kIlp;
    constexpr int NW = ULY_FUSED_CONSUMER_WARPS;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int K = a.stages;
    const int N = int(a.N);
    const FusedSmem L = fused_smem_layout(D, a.N, a.tokens_per_unit, K, a.stage_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kFusedMaxStages;
    float2* turns = reinterpret_cast<float2*>(smem + L.turns);
    int* head_map = reinterpret_cast<int*>(smem + L.heads);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t first = blockIdx.x, step = gridDim.x;
    const int64_t n = first < a.total_units ? (a.total_units - 1 - first) / step + 1 : 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < K; ++s) {
            mbar_init(&full[s], 32);
            mbar_init(&empty[s], NW);
        }
        fence_barrier_init();
    }
    for (int j = threadIdx.x; j < HALF; j += blockDim.x) turns[j] = make_float2(a.turn_hi[j], a.turn_lo[j]);
    for (int g = threadIdx.x; g < N; g += blockDim.x) {
        int r = 0;
        while (r + 1 < a.W && g >= a.head_off[r + 1]) ++r;
        head_map[g] = (r << 16) | int(g - a.head_off[r]);
    }
    __syncthreads();
    if (n == 0) return;
    const int row_bytes = N * D * 2;  // one token, all heads, one tensor

    if (warp == 0) {  // producer
        const uint64_t policy = policy_evict_first();
        int64_t k = 0;
        for (; k < n; ++k) {
            const int s = int(k % K);
            if (k >= K && !mbar_wait_bounded(&empty[s], uint32_t(((k / K) - 1) & 1))) {
                if (lane == 0) atomicOr(&g_fused_status, kStatusWaitTimeout);
                break;
            }
            const FusedUnit t = fused_decode(a, first + k * step);
            float2* table = reinterpret_cast<float2*>(smem + L.tables + s * L.table_bytes);
            const float p0 = float(a.seq_off[t.q] + t.i0);
            for (int e = lane; e < t.ntok * HALF; e += 32) {
                const float2 tj = turns[e % HALF];
                table[e] = rope_cos_sin(p0 + float(e / HALF), tj.x, tj.y);
            }
            __syncwarp();
            if (lane == 0) {
                const uint32_t bytes = uint32_t(t.ntok) * uint32_t(row_bytes);
                const int64_t off = (t.bb * a.s[t.q] + t.i0) * row_bytes;
                uint8_t* dst = smem + L.stages + size_t(s) * a.stage_bytes;
                mbar_arrive_expect_tx(&full[s], 2 * bytes);
                bulk_g2s_hint(dst, a.q_in[t.q] + off, bytes, &full[s], policy);
                bulk_g2s_hint(dst + bytes, a.k_in[t.q] + off, bytes, &full[s], policy);
            } else {
                mbar_arrive(&full[s]);
            }
        }
        // do not leave while copies into this CTA's shared memory are in flight
        if (lane == 0) {
            for (int64_t j = (k > K ? k - K : 0); j < k; ++j) {
                if (!mbar_wait_bounded(&full[j % K], uint32_t((j / K) & 1))) {
                    atomicOr(&g_fused_status, kStatusDrainTimeout);
                    break;
                }
            }
        }
        return;
    }

    // consumers
    const int cw = warp - 1;
    const int sub = lane % G;    // which 8 values of the row this lane holds
    const int group = lane / G;  // which head row of the warp slot
    float wq[8], wk[8];
    {
        const float4* wp = reinterpret_cast<const float4*>(a.rms_w + sub * 8);
        const float4* kp = reinterpret_cast<const float4*>(a.rms_w + D + sub * 8);
        const float4 a0 = wp[0], a1 = wp[1], b0 = kp[0], b1 = kp[1];
        wq[0] = a0.x; wq[1] = a0.y; wq[2] = a0.z; wq[3] = a0.w;
        wq[4] = a1.x; wq[5] = a1.y; wq[6] = a1.z; wq[7] = a1.w;
        wk[0] = b0.x; wk[1] = b0.y; wk[2] = b0.z; wk[3] = b0.w;
        wk[4] = b1.x; wk[5] = b1.y; wk[6] = b1.z; wk[7] = b1.w;
    }
    const float inv_d = 1.0f / float(D);
    const int twoN = 2 * N;
    for (int64_t k = 0; k < n; ++k) {
        const int s = int(k % K);
        const FusedUnit t = fused_decode(a, first + k * step);
        if (!mbar_wait_bounded(&full[s], uint32_t((k / K) & 1))) {
            if (lane == 0) atomicOr(&g_fused_status, kStatusWaitTimeout);
            break;
        }
        const uint8_t* st = smem + L.stages + size_t(s) * a.stage_bytes;
        const float2* table = reinterpret_cast<const float2*>(smem + L.tables + s * L.table_bytes);
        const int items = t.ntok * twoN;  // head rows: (token, q|k, head)
        const int steps = (items + PER_STEP - 1) / PER_STEP;
        const int m_lo = cw * steps / NW, m_hi = (cw + 1) * steps / NW;
        const int64_t row0 = t.bb * a.S + a.seq_off[t.q] + t.i0;  // destination row of token 0
        for (int m = m_lo; m < m_hi; ++m) {
            int tok[kIlp], which[kIlp], head[kIlp];
            bool ok[kIlp];
            float v[kIlp][8], ss[kIlp];
#pragma unroll
            for (int u = 0; u < kIlp; ++u) {
                const int item = m * PER_STEP + u * GPW + group;
                ok[u] = item < items;
                const int it = ok[u] ? item : 0;
                tok[u] = it / twoN;
                const int rem = it - tok[u] * twoN;
                which[u] = rem >= N;
                head[u] = rem - which[u] * N;
                uint4 x = make_uint4(0, 0, 0, 0);
                if (ok[u])
                    x = ld_shared_v4(st + (which[u] * t.ntok + tok[u]) * row_bytes + head[u] * (D * 2) +
                                     sub * 16);
                v[u][0] = bf16_lo(x.x); v[u][1] = bf16_hi(x.x);
                v[u][2] = bf16_lo(x.y); v[u][3] = bf16_hi(x.y);
                v[u][4] = bf16_lo(x.z); v[u][5] = bf16_hi(x.z);
                v[u][6] = bf16_lo(x.w); v[u][7] = bf16_hi(x.w);
                float acc = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc = fmaf(v[u][e], v[u][e], acc);
                ss[u] = acc;
            }
#pragma unroll
            for (int off = G / 2; off > 0; off >>= 1) {
#pragma unroll
                for (int u = 0; u < kIlp; ++u) ss[u] += __shfl_xor_sync(0xffffffffu, ss[u], off);
            }
#pragma unroll
            for (int u = 0; u < kIlp; ++u) {
                if (!ok[u]) continue;
                const float inv = rsqrtf(ss[u] * inv_d + a.eps);
                const float4 cs01 = *reinterpret_cast<const float4*>(table + tok[u] * HALF + sub * 4);
                const float4 cs23 = *reinterpret_cast<const float4*>(table + tok[u] * HALF + sub * 4 + 2);
                const float c[4] = {cs01.x, cs01.z, cs23.x, cs23.z};
                const float sn[4] = {cs01.y, cs01.w, cs23.y, cs23.w};
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float w0 = which[u] ? wk[2 * e] : wq[2 * e];
                    const float w1 = which[u] ? wk[2 * e + 1] : wq[2 * e + 1];
                    const float y0 = v[u][2 * e] * inv * w0;
                    const float y1 = v[u][2 * e + 1] * inv * w1;
                    o[e] = pack_bf16(y0 * c[e] - y1 * sn[e], y0 * sn[e] + y1 * c[e]);
                }
                const int hm = head_map[head[u]];
                const int r = hm >> 16, h = hm & 0xFFFF;
                uint8_t* out = which[u] ? a.k_out[r] : a.q_out[r];
                st_v4(out + ((row0 + tok[u]) * a.n[r] + h) * (D * 2) + sub * 16,
                      make_uint4(o[0], o[1], o[2], o[3]));
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

// Stage geometry for a plan: tokens per unit and stage count (0 stages: does not fit).
void fused_geometry(const Plan& p, int64_t* tokens_per_unit, int* stages, uint32_t* stage_bytes)
{
    *stages = 0;
    *tokens_per_unit = 1;
    *stage_bytes = 0;
    if (p.N > kFusedMaxHeads) return;
    const int64_t pair_bytes = 2 * p.N * p.d * 2;  // one token of q and of k
    int64_t T = ULY_FUSED_STAGE_TARGET / pair_bytes;
    if (T < 1) T = 1;
    const int64_t sb = T * pair_bytes;
    for (int K = kFusedMaxStages; K >= 2; --K) {
        const FusedSmem m = fused_smem_layout(int(p.d), p.N, int(T), K, uint32_t(sb));
        if (sb <= (1 << 20) && m.total <= kFusedSmemBudget) {
            *tokens_per_unit = T;
            *stages = K;
            *stage_bytes = uint32_t(sb);
            return;
        }
    }
}

static int g_fused_smem_set[64];

template <int G>
static cudaError_t launch_g(const FusedArgs& a, cudaStream_t stream, int device, int grid)
{
    constexpr int bit = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : G == 8 ? 3 : G == 16 ? 4 : 5;
    if (device >= 0 && device < 64 && !(g_fused_smem_set[device] & (1 << bit))) {
        cudaError_t e = cudaFuncSetAttribute(fused_qk_kernel<G>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kFusedSmemBudget);
        if (e != cudaSuccess) return e;
        g_fused_smem_set[device] |= 1 << bit;
    }
    const FusedSmem m = fused_smem_layout(a.d, a.N, a.tokens_per_unit, a.stages, a.stage_bytes);
    fused_qk_kernel<G><<<grid, kFusedThreads, m.total, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t fused_launch(const FusedArgs& a, cudaStream_t stream, int device, int sm_count)
{
    if (a.total_units == 0) return cudaSuccess;
    int64_t grid = sm_count;
    if (grid > a.total_units) grid = a.total_units;
    switch (a.d / 8) {
        case 1: return launch_g<1>(a, stream, device, int(grid));
        case 2: return launch_g<2>(a, stream, device, int(grid));
        case 4: return launch_g<4>(a, stream, device, int(grid));
        case 8: return launch_g<8>(a, stream, device, int(grid));
        case 16: return launch_g<16>(a, stream, device, int(grid));
        case 32: return launch_g<32>(a, stream, device, int(grid));
        default: return cudaErrorInvalidValue;
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
