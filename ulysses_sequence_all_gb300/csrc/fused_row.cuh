// fused_row.cuh -- how a lane group of the fused kernels holds one head row: the element type
// (bf16 or fp16) and the RoPE pair layout (adjacent pairs (2j, 2j+1), or rotate-half pairs
// (j, j + d/2)), both with the angle p * theta^(-2j/d) for pair j.
//
// A lane holds P of the row's RoPE pairs and a group of G = d / (2P) lanes holds a row. The pairs
// sit in registers as packed float2 values: fst[h] holds the first elements of two of the lane's
// pairs, snd[h] their second elements (h < P / 2), so the rotation, the weights and the cos/sin
// table are the same code for every layout. The layouts (WIDE selects P = 8 where d >= 16):
//  * adjacent, P = 4: the lane's pairs are j = 4 sub .. 4 sub + 3, elements 8 sub .. 8 sub + 7,
//    one 16-byte word;
//  * adjacent, P = 8: two such words, one in each half of the row: pairs 4 sub .. 4 sub + 3 and
//    d/4 + 4 sub .. d/4 + 4 sub + 3 (16 bytes at byte 16 sub and at byte d + 16 sub);
//  * rotate half, P = 8 (always used for d >= 16): pairs j = 8 sub .. 8 sub + 7, first elements
//    8 sub .. 8 sub + 7 (16 bytes at byte 16 sub) and second elements d/2 + 8 sub .. d/2 +
//    8 sub + 7 (16 bytes at byte d + 16 sub);
//  * rotate half, d = 8 (P = 4): 8 bytes of each half.
// Every layout moves a lane's bytes with 16-byte shared-memory accesses (d = 8 aside), 8 lanes of
// a quarter warp covering 128 contiguous bytes, so the accesses are free of bank conflicts. A
// row's raw form is P 32-bit words (two elements each), in the order the lane loads them.
// Head dimensions that are not powers of two (any multiple of 8 up to 256) use the same layouts
// with d read at run time (RowIO<..., D < 8, ...> below): P = 8 where 16 divides d, else P = 4;
// G = d / (2P) lanes per row then need not divide the warp (row_lane_stride).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace uly {

// Position in a ring of K shared-memory stages: the stage of the current unit and the parity of
// its use (unit j uses stage j mod K for the (j div K)-th time), advanced without division.
struct StageRing {
    int s = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next(int K)
    {
        if (++s == K) {
            s = 0;
            phase ^= 1u;
        }
    }
};

// cos and sin of 2 pi * frac(p * (hi + lo)), p a non-negative integer below 2^24: the angle in
// turns, with p * hi split exactly into a product and its fma residual (an error-free product),
// the whole turns dropped (exact), then the small terms added.
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

template <bool F16>
struct ElemT;

template <>
struct ElemT<false> {  // bf16: the upper half of a binary32
    static __device__ __forceinline__ float lo(uint32_t w) { return __uint_as_float(w << 16); }
    static __device__ __forceinline__ float hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
    static __device__ __forceinline__ uint32_t pack(float l, float h)
    {
        const __nv_bfloat162 v = __floats2bfloat162_rn(l, h);  // round to nearest even
        return *reinterpret_cast<const uint32_t*>(&v);
    }
};

template <>
struct ElemT<true> {  // IEEE binary16
    static __device__ __forceinline__ float lo(uint32_t w)
    {
        return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
    }
    static __device__ __forceinline__ float hi(uint32_t w)
    {
        return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
    }
    static __device__ __forceinline__ uint32_t pack(float l, float h)
    {
        const __half2 v = __floats2half2_rn(l, h);  // round to nearest even
        return *reinterpret_cast<const uint32_t*>(&v);
    }
};

// A row's head dimension and lanes, for the layouts whose head dimension is known only at run
// time (RowIO<..., 0, ...>); the compile-time layouts take and ignore it.
struct RowDims {
    int d;  // head dimension
    int g;  // lanes holding the row's pairs
};

template <bool F16, bool HALF, int D, bool WIDE = false>
struct RowIO {
    using E = ElemT<F16>;
    static constexpr int P = ((HALF || WIDE) && D >= 16) ? 8 : 4;  // pairs per lane
    static constexpr int H = P / 2;                               // float2 slots per lane and kind
    static constexpr int G = D / (2 * P);                         // lanes per row
    static_assert(G >= 1 && 32 % G == 0, "a row's lanes must divide a warp");
    struct Words {
        uint32_t w[P];
    };
    static __device__ __forceinline__ constexpr RowDims dims(int) { return RowDims{D, G}; }

    // The lane's raw words of the row starting at `row` (shared memory).
    static __device__ __forceinline__ Words load(const uint8_t* row, int sub)
    {
        Words r;
        if constexpr (!HALF && P == 4) {
            const uint4 a = ld_shared_v4(row + sub * 16);
            r.w[0] = a.x, r.w[1] = a.y, r.w[2] = a.z, r.w[3] = a.w;
        } else if constexpr (P == 4) {
            const uint2 a = ld_shared_v2(row + sub * 8);
            const uint2 b = ld_shared_v2(row + D + sub * 8);
            r.w[0] = a.x, r.w[1] = a.y, r.w[2] = b.x, r.w[3] = b.y;
        } else {
            const uint4 a = ld_shared_v4(row + sub * 16);
            const uint4 b = ld_shared_v4(row + D + sub * 16);
            r.w[0] = a.x, r.w[1] = a.y, r.w[2] = a.z, r.w[3] = a.w;
            r.w[4] = b.x, r.w[5] = b.y, r.w[6] = b.z, r.w[7] = b.w;
        }
        return r;
    }

    static __device__ __forceinline__ void store(uint8_t* row, int sub, const Words& r)
    {
        if constexpr (!HALF && P == 4) {
            st_shared_v4(row + sub * 16, make_uint4(r.w[0], r.w[1], r.w[2], r.w[3]));
        } else if constexpr (P == 4) {
            st_shared_v2(row + sub * 8, r.w[0], r.w[1]);
            st_shared_v2(row + D + sub * 8, r.w[2], r.w[3]);
        } else {
            st_shared_v4(row + sub * 16, make_uint4(r.w[0], r.w[1], r.w[2], r.w[3]));
            st_shared_v4(row + D + sub * 16, make_uint4(r.w[4], r.w[5], r.w[6], r.w[7]));
        }
    }

    // The lane's raw words to the row starting at `row` in global memory.
    static __device__ __forceinline__ void store_global(uint8_t* row, int sub, const Words& r)
    {
        if constexpr (!HALF && P == 4) {
            st_v4(row + sub * 16, make_uint4(r.w[0], r.w[1], r.w[2], r.w[3]));
        } else if constexpr (P == 4) {
            st_v2(row + sub * 8, r.w[0], r.w[1]);
            st_v2(row + D + sub * 8, r.w[2], r.w[3]);
        } else {
            st_v4(row + sub * 16, make_uint4(r.w[0], r.w[1], r.w[2], r.w[3]));
            st_v4(row + D + sub * 16, make_uint4(r.w[4], r.w[5], r.w[6], r.w[7]));
        }
    }

    // raw words -> first / second elements of the lane's pairs P sub + 2h, P sub + 2h + 1
    static __device__ __forceinline__ void unpack(const Words& r, int h, float2& fst, float2& snd)
    {
        if constexpr (!HALF) {
            const uint32_t w0 = r.w[2 * h], w1 = r.w[2 * h + 1];
            fst = make_float2(E::lo(w0), E::lo(w1));
            snd = make_float2(E::hi(w0), E::hi(w1));
        } else {
            const uint32_t f = r.w[h], s = r.w[H + h];
            fst = make_float2(E::lo(f), E::hi(f));
            snd = make_float2(E::lo(s), E::hi(s));
        }
    }

    // first / second elements (rounded once to the element type) -> raw words
    static __device__ __forceinline__ Words pack(const float2 fst[H], const float2 snd[H])
    {
        Words r;
#pragma unroll
        for (int h = 0; h < H; ++h) {
            if constexpr (!HALF) {
                r.w[2 * h] = E::pack(fst[h].x, snd[h].x);
                r.w[2 * h + 1] = E::pack(fst[h].y, snd[h].y);
            } else {
                r.w[h] = E::pack(fst[h].x, fst[h].y);
                r.w[H + h] = E::pack(snd[h].x, snd[h].y);
            }
        }
        return r;
    }

    // Column (element index in the row) of fst[h] (second = false) or snd[h], component k.
    static __device__ __forceinline__ constexpr int col(int sub, int h, bool second, int k)
    {
        return HALF ? (second ? D / 2 : 0) + P * sub + 2 * h + k
                    : (h >= 2 ? D / 2 : 0) + 8 * sub + 4 * (h & 1) + 2 * k + (second ? 1 : 0);
    }

    // Index of the float4 table entry (c_j, c_j+1, s_j, s_j+1), j = P sub + 2h, of token tok.
    static __device__ __forceinline__ constexpr int table_entry(int tok, int h, int sub)
    {
        return (tok * H + h) * G + sub;
    }

    // Float offset of pair jj's cosine in a token table (its sine is 2 floats further): the
    // entry of the lane that holds the pair, component jj & 1.
    static __device__ __forceinline__ constexpr int table_at(int tok, int jj)
    {
        if constexpr (HALF || P == 4) {  // the lane's pairs are P consecutive ones
            return table_entry(tok, (jj % P) >> 1, jj / P) * 4 + (jj & 1);
        } else {  // chunk c = jj / (d/4) of the row; 4 pairs per lane in each chunk
            const int c = jj / (D / 4), jr = jj % (D / 4);
            return table_entry(tok, 2 * c + ((jr & 3) >> 1), jr >> 2) * 4 + (jj & 1);
        }
    }

    // The lane's weights in the same arrangement (w: d fp32 values, 16-byte aligned).
    static __device__ __forceinline__ void weights(const float* w, int sub, float2 fst[H],
                                                   float2 snd[H])
    {
        if constexpr (!HALF) {
#pragma unroll
            for (int c = 0; c < P / 4; ++c) {  // the lane's chunk in each half of the row
                const float4 a0 = *reinterpret_cast<const float4*>(w + c * (D / 2) + 8 * sub);
                const float4 a1 = *reinterpret_cast<const float4*>(w + c * (D / 2) + 8 * sub + 4);
                fst[2 * c] = make_float2(a0.x, a0.z);
                snd[2 * c] = make_float2(a0.y, a0.w);
                fst[2 * c + 1] = make_float2(a1.x, a1.z);
                snd[2 * c + 1] = make_float2(a1.y, a1.w);
            }
        } else {
#pragma unroll
            for (int q = 0; q < P / 4; ++q) {
                const float4 f = *reinterpret_cast<const float4*>(w + P * sub + 4 * q);
                const float4 s = *reinterpret_cast<const float4*>(w + D / 2 + P * sub + 4 * q);
                fst[2 * q] = make_float2(f.x, f.y);
                fst[2 * q + 1] = make_float2(f.z, f.w);
                snd[2 * q] = make_float2(s.x, s.y);
                snd[2 * q + 1] = make_float2(s.z, s.w);
            }
        }
    }

    // The same, in the form the run-time layouts take (the dimensions are this layout's own).
    static __device__ __forceinline__ Words load(const uint8_t* row, int sub, RowDims)
    {
        return load(row, sub);
    }
    static __device__ __forceinline__ void store(uint8_t* row, int sub, const Words& r, RowDims)
    {
        store(row, sub, r);
    }
    static __device__ __forceinline__ void store_global(uint8_t* row, int sub, const Words& r,
                                                        RowDims)
    {
        store_global(row, sub, r);
    }
    static __device__ __forceinline__ constexpr int col(int sub, int h, bool second, int k, RowDims)
    {
        return col(sub, h, second, k);
    }
    static __device__ __forceinline__ constexpr int table_entry(int tok, int h, int sub, RowDims)
    {
        return table_entry(tok, h, sub);
    }
    static __device__ __forceinline__ constexpr int table_at(int tok, int jj, RowDims)
    {
        return table_at(tok, jj);
    }
    static __device__ __forceinline__ void weights(const float* w, int sub, float2 fst[H],
                                                   float2 snd[H], RowDims)
    {
        weights(w, sub, fst, snd);
    }
};

// Head dimension known at run time: D below 8 selects one of four layouts, all with d read at run
// time and any d that is a multiple of 8 (a head row of 2-byte elements is a whole number of
// 16-byte words): bit 0 set, eight pairs per lane (d a multiple of 16), else four; the layouts are
// those above for P = 8 and P = 4. A row takes g = d / (2 P) lanes, which need not divide the
// warp. Bit 1 set: rows start on power-of-two lane boundaries (g rounded up), reduced with a
// butterfly; clear: rows packed back to back, floor(32 / g) of them, reduced towards their first
// lane. The host takes the packed form only where it fits more rows in a warp (row_lane_stride).
constexpr int kRtWide = 1, kRtPow2 = 2;
__host__ __device__ constexpr bool rt_layout(int D) { return D < 8; }
__host__ __device__ constexpr bool rt_pow2(int D) { return D >= 8 || (D & kRtPow2) != 0; }

template <bool F16, bool HALF, int PP>
struct RowIORt {
    using E = ElemT<F16>;
    static constexpr int P = PP;
    static constexpr int H = P / 2;
    static constexpr int G = 0;  // run time: RowDims::g
    struct Words {
        uint32_t w[P];
    };
    static __device__ __forceinline__ constexpr RowDims dims(int d) { return RowDims{d, d / (2 * P)}; }

    static __device__ __forceinline__ Words load(const uint8_t* row, int sub, RowDims r)
    {
        Words x;
        if constexpr (!HALF && P == 4) {
            const uint4 a = ld_shared_v4(row + sub * 16);
            x.w[0] = a.x, x.w[1] = a.y, x.w[2] = a.z, x.w[3] = a.w;
        } else if constexpr (P == 4) {
            const uint2 a = ld_shared_v2(row + sub * 8);
            const uint2 b = ld_shared_v2(row + r.d + sub * 8);
            x.w[0] = a.x, x.w[1] = a.y, x.w[2] = b.x, x.w[3] = b.y;
        } else {
            const uint4 a = ld_shared_v4(row + sub * 16);
            const uint4 b = ld_shared_v4(row + r.d + sub * 16);
            x.w[0] = a.x, x.w[1] = a.y, x.w[2] = a.z, x.w[3] = a.w;
            x.w[4] = b.x, x.w[5] = b.y, x.w[6] = b.z, x.w[7] = b.w;
        }
        return x;
    }

    static __device__ __forceinline__ void store(uint8_t* row, int sub, const Words& x, RowDims r)
    {
        if constexpr (!HALF && P == 4) {
            st_shared_v4(row + sub * 16, make_uint4(x.w[0], x.w[1], x.w[2], x.w[3]));
        } else if constexpr (P == 4) {
            st_shared_v2(row + sub * 8, x.w[0], x.w[1]);
            st_shared_v2(row + r.d + sub * 8, x.w[2], x.w[3]);
        } else {
            st_shared_v4(row + sub * 16, make_uint4(x.w[0], x.w[1], x.w[2], x.w[3]));
            st_shared_v4(row + r.d + sub * 16, make_uint4(x.w[4], x.w[5], x.w[6], x.w[7]));
        }
    }

    static __device__ __forceinline__ void store_global(uint8_t* row, int sub, const Words& x,
                                                        RowDims r)
    {
        if constexpr (!HALF && P == 4) {
            st_v4(row + sub * 16, make_uint4(x.w[0], x.w[1], x.w[2], x.w[3]));
        } else if constexpr (P == 4) {
            st_v2(row + sub * 8, x.w[0], x.w[1]);
            st_v2(row + r.d + sub * 8, x.w[2], x.w[3]);
        } else {
            st_v4(row + sub * 16, make_uint4(x.w[0], x.w[1], x.w[2], x.w[3]));
            st_v4(row + r.d + sub * 16, make_uint4(x.w[4], x.w[5], x.w[6], x.w[7]));
        }
    }

    static __device__ __forceinline__ void unpack(const Words& x, int h, float2& fst, float2& snd)
    {
        if constexpr (!HALF) {
            const uint32_t w0 = x.w[2 * h], w1 = x.w[2 * h + 1];
            fst = make_float2(E::lo(w0), E::lo(w1));
            snd = make_float2(E::hi(w0), E::hi(w1));
        } else {
            const uint32_t f = x.w[h], s = x.w[H + h];
            fst = make_float2(E::lo(f), E::hi(f));
            snd = make_float2(E::lo(s), E::hi(s));
        }
    }

    static __device__ __forceinline__ Words pack(const float2 fst[H], const float2 snd[H])
    {
        Words x;
#pragma unroll
        for (int h = 0; h < H; ++h) {
            if constexpr (!HALF) {
                x.w[2 * h] = E::pack(fst[h].x, snd[h].x);
                x.w[2 * h + 1] = E::pack(fst[h].y, snd[h].y);
            } else {
                x.w[h] = E::pack(fst[h].x, fst[h].y);
                x.w[H + h] = E::pack(snd[h].x, snd[h].y);
            }
        }
        return x;
    }

    static __device__ __forceinline__ constexpr int col(int sub, int h, bool second, int k,
                                                        RowDims r)
    {
        return HALF ? (second ? r.d / 2 : 0) + P * sub + 2 * h + k
                    : (h >= 2 ? r.d / 2 : 0) + 8 * sub + 4 * (h & 1) + 2 * k + (second ? 1 : 0);
    }

    static __device__ __forceinline__ constexpr int table_entry(int tok, int h, int sub, RowDims r)
    {
        return (tok * H + h) * r.g + sub;
    }

    static __device__ __forceinline__ int table_at(int tok, int jj, RowDims r)
    {
        if constexpr (HALF || P == 4) {
            return table_entry(tok, (jj % P) >> 1, jj / P, r) * 4 + (jj & 1);
        } else {  // chunk c = jj / (d/4) of the row; 4 pairs per lane in each chunk
            const int q4 = r.d / 4, c = jj >= q4, jr = jj - c * q4;
            return table_entry(tok, 2 * c + ((jr & 3) >> 1), jr >> 2, r) * 4 + (jj & 1);
        }
    }

    static __device__ __forceinline__ void weights(const float* w, int sub, float2 fst[H],
                                                   float2 snd[H], RowDims r)
    {
        if constexpr (!HALF) {
#pragma unroll
            for (int c = 0; c < P / 4; ++c) {  // the lane's chunk in each half of the row
                const float4 a0 = *reinterpret_cast<const float4*>(w + c * (r.d / 2) + 8 * sub);
                const float4 a1 = *reinterpret_cast<const float4*>(w + c * (r.d / 2) + 8 * sub + 4);
                fst[2 * c] = make_float2(a0.x, a0.z);
                snd[2 * c] = make_float2(a0.y, a0.w);
                fst[2 * c + 1] = make_float2(a1.x, a1.z);
                snd[2 * c + 1] = make_float2(a1.y, a1.w);
            }
        } else {
#pragma unroll
            for (int q = 0; q < P / 4; ++q) {
                const float4 f = *reinterpret_cast<const float4*>(w + P * sub + 4 * q);
                const float4 s = *reinterpret_cast<const float4*>(w + r.d / 2 + P * sub + 4 * q);
                fst[2 * q] = make_float2(f.x, f.y);
                fst[2 * q + 1] = make_float2(f.z, f.w);
                snd[2 * q] = make_float2(s.x, s.y);
                snd[2 * q + 1] = make_float2(s.z, s.w);
            }
        }
    }
};

template <bool F16, bool HALF, bool WIDE>
struct RowIO<F16, HALF, 0, WIDE> : RowIORt<F16, HALF, 4> {};
template <bool F16, bool HALF, bool WIDE>
struct RowIO<F16, HALF, kRtWide, WIDE> : RowIORt<F16, HALF, 8> {};
template <bool F16, bool HALF, bool WIDE>
struct RowIO<F16, HALF, kRtPow2, WIDE> : RowIORt<F16, HALF, 4> {};
template <bool F16, bool HALF, bool WIDE>
struct RowIO<F16, HALF, kRtPow2 | kRtWide, WIDE> : RowIORt<F16, HALF, 8> {};

// Lanes from one row's first lane to the next row's in a warp, for a row of g lanes (g <= 32):
// g rounded up to a power of two when that leaves as many rows in the warp (rows then sit on
// power-of-two lane boundaries and reduce with a butterfly), else g itself (rows packed back to
// back, more of them per warp, reduced lane by lane).
__host__ __device__ inline int row_lane_stride(int g)
{
    int p = 1;
    while (p < g) p <<= 1;
    return 32 / p == 32 / g ? p : g;
}

// The run-time layout (D < 8) for head dimension d.
inline int rt_layout_for(int d)
{
    const bool wide = d % 16 == 0;
    const int g = d / (wide ? 16 : 8);
    const int gp = row_lane_stride(g);
    return (wide ? kRtWide : 0) | ((gp & (gp - 1)) == 0 ? kRtPow2 : 0);
}

// Sums of v[u] and w[u] (K = 1: v only) over the g lanes of one row (lanes group * gp + 0 ..
// g - 1), in every one of them; lanes of the group past g hold zeros. Rows on power-of-two lane
// strides (rt_pow2(D)): a butterfly over gp lanes; else a reduction towards the row's first lane,
// then a broadcast from it.
template <int D, int K, int N>
__device__ __forceinline__ void row_sums(float (&v)[N], float (&w)[N], int g, int gp, int sub,
                                         int group)
{
    if constexpr (rt_pow2(D)) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            if (off >= gp) continue;
#pragma unroll
            for (int u = 0; u < N; ++u) {
                v[u] += __shfl_xor_sync(0xffffffffu, v[u], off);
                if constexpr (K == 2) w[u] += __shfl_xor_sync(0xffffffffu, w[u], off);
            }
        }
    } else {
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            if (off >= g) break;
#pragma unroll
            for (int u = 0; u < N; ++u) {
                const float t = __shfl_down_sync(0xffffffffu, v[u], off);
                if (sub + off < g) v[u] += t;
                if constexpr (K == 2) {
                    const float t2 = __shfl_down_sync(0xffffffffu, w[u], off);
                    if (sub + off < g) w[u] += t2;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < N; ++u) {
            v[u] = __shfl_sync(0xffffffffu, v[u], group * gp);
            if constexpr (K == 2) w[u] = __shfl_sync(0xffffffffu, w[u], group * gp);
        }
    }
}

}  // namespace uly
