// fused_qk.cu -- mode-0 relayout of q and k with QK RMSNorm + RoPE applied in the scatter
// (fast-ulysses 0.1.0, "Fusion examples": QK RMSNorm + RoPE inside the scatter kernel).
//
// Per head row x of d bf16 values at global sequence position p:
//     y = x / sqrt(mean(x^2) + eps) * w,   (y[2j], y[2j+1]) rotated by p * theta^(-2j/d),
// in fp32, rounded once to bf16 (nearest even), and written where mode 0 places the row.
//
// Structure: a persistent grid with one CTA per SM. Warp 0 is the producer: one lane streams
// work units (a few consecutive tokens of one source rank: all N heads of q and of k, two
// contiguous spans) into a ring of shared-memory stages with cp.async.bulk, completing on the
// stage's "full" mbarrier. The consumer warps split a stage's head rows among themselves in
// contiguous ranges; a group of d/8 lanes holds one head row (8 values per lane), reduces the sum
// of squares with xor shuffles, applies the weight and the rotation, and stores 16 bytes per lane
// straight to the destination rank (each head row is one contiguous 2d-byte span there). Each
// consumer warp then arrives on the stage's "empty" mbarrier so the producer can refill it.
//
// RoPE angles: p * theta^(-2j/d) reaches ~75,600 rad at the Wan shape, where an fp32 product
// alone is off by ~5e-3 rad. The angle is instead formed in turns (units of 2 pi): the host
// supplies theta^(-2j/d) / (2 pi) as a float pair hi + lo, the kernel forms p * hi exactly as a
// product plus its fma residual, drops the integer part (exact), adds the small terms, and calls
// sincospif on the reduced fraction; the angle error stays near 1e-6 rad.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/ulysses.h"
#include "plan.h"
#include "ptx.cuh"

namespace uly {

static __device__ unsigned g_fused_status;

#ifndef ULY_FUSED_CONSUMER_WARPS
#define ULY_FUSED_CONSUMER_WARPS 8
#endif
#ifndef ULY_FUSED_STAGE_TARGET
#define ULY_FUSED_STAGE_TARGET 40960
#endif
constexpr int kFusedMaxStages = 6;
constexpr int kFusedSmemBudget = 200 * 1024;
constexpr int kFusedHeader = 128;  // 2 * kFusedMaxStages barriers
constexpr int kFusedThreads = 32 * (1 + ULY_FUSED_CONSUMER_WARPS);

struct FusedUnit {
    int q;
    int64_t bb, i0, ntok;
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
    t.ntok = min(T, rows - blk * T);
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
__device__ __forceinline__ void rope_cos_sin(float p, float hi, float lo, float* c, float* s)
{
    const float ph = p * hi;
    const float pe = fmaf(p, hi, -ph);  // exact residual of the product
    float f = ph - rintf(ph);           // exact: drops whole turns
    f += fmaf(p, lo, pe);
    sincospif(2.0f * f, s, c);
}

template <int G>  // lanes per head row; d = 8 * G
__global__ void __launch_bounds__(kFusedThreads, 1) fused_qk_kernel(const __grid_constant__ FusedArgs a)
{
    constexpr int D = 8 * G;
    constexpr int GPW = 32 / G;  // head rows per warp step
    constexpr int NW = ULY_FUSED_CONSUMER_WARPS;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kFusedMaxStages;
    uint8_t* stage0 = smem + kFusedHeader;
    const int K = a.stages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t first = blockIdx.x, step = gridDim.x;
    const int64_t n = first < a.total_units ? (a.total_units - 1 - first) / step + 1 : 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < K; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        fence_barrier_init();
    }
    __syncthreads();
    if (n == 0) return;
    const int64_t row_bytes = a.N * D * 2;  // one token, all heads, one tensor

    if (warp == 0) {  // producer
        if (lane != 0) return;
        const uint64_t policy = policy_evict_first();
        int64_t k = 0;
        for (; k < n; ++k) {
            const int s = int(k % K);
            if (k >= K && !mbar_wait_bounded(&empty[s], uint32_t(((k / K) - 1) & 1))) {
                atomicOr(&g_fused_status, kStatusWaitTimeout);
                break;
            }
            const FusedUnit t = fused_decode(a, first + k * step);
            const uint32_t bytes = uint32_t(t.ntok * row_bytes);
            const int64_t off = (t.bb * a.s[t.q] + t.i0) * row_bytes;
            uint8_t* dst = stage0 + size_t(s) * a.stage_bytes;
            mbar_arrive_expect_tx(&full[s], 2 * bytes);
            bulk_g2s_hint(dst, a.q_in[t.q] + off, bytes, &full[s], policy);
            bulk_g2s_hint(dst + bytes, a.k_in[t.q] + off, bytes, &full[s], policy);
        }
        // do not leave while copies into this CTA's shared memory are in flight
        for (int64_t j = (k > K ? k - K : 0); j < k; ++j) {
            if (!mbar_wait_bounded(&full[j % K], uint32_t((j / K) & 1))) {
                atomicOr(&g_fused_status, kStatusDrainTimeout);
                break;
            }
        }
        return;
    }

    // consumers
    const int cw = warp - 1;
    const int sub = lane % G;   // which 8 values of the row this lane holds
    const int group = lane / G; // which head row of the warp step
    float wq[8], wk[8], th[4], tl[4];
    {
        const float4* wp = reinterpret_cast<const float4*>(a.rms_w + sub * 8);
        const float4* kp = reinterpret_cast<const float4*>(a.rms_w + D + sub * 8);
        const float4 a0 = wp[0], a1 = wp[1], b0 = kp[0], b1 = kp[1];
        wq[0] = a0.x; wq[1] = a0.y; wq[2] = a0.z; wq[3] = a0.w;
        wq[4] = a1.x; wq[5] = a1.y; wq[6] = a1.z; wq[7] = a1.w;
        wk[0] = b0.x; wk[1] = b0.y; wk[2] = b0.z; wk[3] = b0.w;
        wk[4] = b1.x; wk[5] = b1.y; wk[6] = b1.z; wk[7] = b1.w;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            th[m] = a.turn_hi[sub * 4 + m];
            tl[m] = a.turn_lo[sub * 4 + m];
        }
    }
    const float inv_d = 1.0f / float(D);
    const int64_t N = a.N;
    for (int64_t k = 0; k < n; ++k) {
        const int s = int(k % K);
        const FusedUnit t = fused_decode(a, first + k * step);
        if (!mbar_wait_bounded(&full[s], uint32_t((k / K) & 1))) {
            if (lane == 0) atomicOr(&g_fused_status, kStatusWaitTimeout);
            break;
        }
        const uint8_t* st = stage0 + size_t(s) * a.stage_bytes;
        const int64_t items = 2 * t.ntok * N;  // head rows: (token, q|k, head)
        const int64_t steps = (items + GPW - 1) / GPW;
        const int64_t m_lo = cw * steps / NW, m_hi = (cw + 1) * steps / NW;
        int64_t cur_tok = -1;
        float cs[4], sn[4];
        for (int64_t m = m_lo; m < m_hi; ++m) {
            const int64_t item = m * GPW + group;
            const bool valid = item < items;
            const int64_t tok = valid ? item / (2 * N) : 0;
            const int64_t rem = item - tok * 2 * N;
            const int which = valid && rem >= N;  // 0: q, 1: k
            const int64_t head = valid ? rem - which * N : 0;
            uint4 x = make_uint4(0, 0, 0, 0);
            if (valid)
                x = ld_shared_v4(st + (which * t.ntok + tok) * row_bytes + head * (D * 2) + sub * 16);
            float v[8] = {bf16_lo(x.x), bf16_hi(x.x), bf16_lo(x.y), bf16_hi(x.y),
                          bf16_lo(x.z), bf16_hi(x.z), bf16_lo(x.w), bf16_hi(x.w)};
            float ss = 0.f;
#pragma unroll
            for (int m2 = 0; m2 < 8; ++m2) ss = fmaf(v[m2], v[m2], ss);
#pragma unroll
            for (int off = G / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            if (!valid) continue;
            if (tok != cur_tok) {
                const float p = float(a.seq_off[t.q] + t.i0 + tok);
#pragma unroll
                for (int m2 = 0; m2 < 4; ++m2) rope_cos_sin(p, th[m2], tl[m2], &cs[m2], &sn[m2]);
                cur_tok = tok;
            }
            const float inv = rsqrtf(ss * inv_d + a.eps);
            uint32_t o[4];
#pragma unroll
            for (int m2 = 0; m2 < 4; ++m2) {
                const float y0 = v[2 * m2] * inv * (which ? wk[2 * m2] : wq[2 * m2]);
                const float y1 = v[2 * m2 + 1] * inv * (which ? wk[2 * m2 + 1] : wq[2 * m2 + 1]);
                o[m2] = pack_bf16(y0 * cs[m2] - y1 * sn[m2], y0 * sn[m2] + y1 * cs[m2]);
            }
            int r = 0;
            while (r + 1 < a.W && head >= a.head_off[r + 1]) ++r;
            const int64_t h = head - a.head_off[r];
            uint8_t* out = which ? a.k_out[r] : a.q_out[r];
            uint8_t* dst = out + ((t.bb * a.S + a.seq_off[t.q] + t.i0 + tok) * a.n[r] + h) * (D * 2) +
                           sub * 16;
            st_v4(dst, make_uint4(o[0], o[1], o[2], o[3]));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

// Stage geometry for a plan: tokens per unit and stage count (0 stages: the row is too wide).
void fused_geometry(const Plan& p, int64_t* tokens_per_unit, int* stages, uint32_t* stage_bytes)
{
    const int64_t pair_bytes = 2 * p.N * p.d * 2;  // one token of q and of k
    int64_t T = ULY_FUSED_STAGE_TARGET / pair_bytes;
    if (T < 1) T = 1;
    const int64_t sb = T * pair_bytes;
    int64_t K = (kFusedSmemBudget - kFusedHeader) / sb;
    if (K > kFusedMaxStages) K = kFusedMaxStages;
    *tokens_per_unit = T;
    *stages = K >= 2 ? int(K) : 0;
    *stage_bytes = uint32_t(sb);
}

static int g_fused_smem_set[64];

template <int G>
static cudaError_t launch_g(const FusedArgs& a, cudaStream_t stream, int device, int grid, int smem)
{
    constexpr int bit = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : G == 8 ? 3 : G == 16 ? 4 : 5;
    if (device >= 0 && device < 64 && !(g_fused_smem_set[device] & (1 << bit))) {
        cudaError_t e = cudaFuncSetAttribute(fused_qk_kernel<G>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kFusedSmemBudget);
        if (e != cudaSuccess) return e;
        g_fused_smem_set[device] |= 1 << bit;
    }
    fused_qk_kernel<G><<<grid, kFusedThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t fused_launch(const FusedArgs& a, cudaStream_t stream, int device, int sm_count)
{
    if (a.total_units == 0) return cudaSuccess;
    int64_t grid = sm_count;
    if (grid > a.total_units) grid = a.total_units;
    const int smem = kFusedHeader + a.stages * int(a.stage_bytes);
    switch (a.d / 8) {
        case 1: return launch_g<1>(a, stream, device, int(grid), smem);
        case 2: return launch_g<2>(a, stream, device, int(grid), smem);
        case 4: return launch_g<4>(a, stream, device, int(grid), smem);
        case 8: return launch_g<8>(a, stream, device, int(grid), smem);
        case 16: return launch_g<16>(a, stream, device, int(grid), smem);
        case 32: return launch_g<32>(a, stream, device, int(grid), smem);
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
