// fused_row.cuh -- how a lane group of the fused kernels holds one head row: the element type
// (bf16 or fp16) and the RoPE pair layout (adjacent pairs (2j, 2j+1), or rotate-half pairs
// (j, j + d/2)), both with the angle p * theta^(-2j/d) for pair j.
//
// A group of d/8 lanes holds a row. In both layouts lane `sub` works on pairs j = 4 sub ..
// 4 sub + 3, as packed float2 values: fst[h] holds the first elements of pairs 4 sub + 2h and
// 4 sub + 2h + 1, snd[h] their second elements (h = 0, 1), so the rotation, the weights and the
// cos/sin table are the same code for both layouts:
//  * adjacent: the lane's pairs are elements 8 sub .. 8 sub + 7, one 16-byte word;
//  * rotate half: first elements 4 sub .. 4 sub + 3 (8 bytes at byte 8 sub) and second elements
//    d/2 + 4 sub .. d/2 + 4 sub + 3 (8 bytes at byte d + 8 sub).
// A row's raw form is four 32-bit words (two elements each): the 16-byte word (adjacent), or the
// first-half then the second-half 8 bytes (rotate half).
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

template <bool F16, bool HALF, int D>
struct RowIO {
    using E = ElemT<F16>;

    // The lane's four raw words of the row starting at `row` (shared memory).
    static __device__ __forceinline__ uint4 load(const uint8_t* row, int sub)
    {
        if constexpr (!HALF) {
            return ld_shared_v4(row + sub * 16);
        } else {
            const uint2 a = ld_shared_v2(row + sub * 8);
            const uint2 b = ld_shared_v2(row + D + sub * 8);
            return make_uint4(a.x, a.y, b.x, b.y);
        }
    }

    static __device__ __forceinline__ void store(uint8_t* row, int sub, const uint4& w)
    {
        if constexpr (!HALF) {
            st_shared_v4(row + sub * 16, w);
        } else {
            st_shared_v2(row + sub * 8, w.x, w.y);
            st_shared_v2(row + D + sub * 8, w.z, w.w);
        }
    }

    // raw words -> first / second elements of the lane's pairs, h = 0, 1
    static __device__ __forceinline__ void unpack(const uint4& w, int h, float2& fst, float2& snd)
    {
        const uint32_t w0 = h ? w.z : w.x, w1 = h ? w.w : w.y;
        if constexpr (!HALF) {
            fst = make_float2(E::lo(w0), E::lo(w1));
            snd = make_float2(E::hi(w0), E::hi(w1));
        } else {
            const uint32_t f = h ? w.y : w.x, s = h ? w.w : w.z;
            fst = make_float2(E::lo(f), E::hi(f));
            snd = make_float2(E::lo(s), E::hi(s));
        }
    }

    // first / second elements (rounded once to the element type) -> raw words
    static __device__ __forceinline__ uint4 pack(const float2 fst[2], const float2 snd[2])
    {
        if constexpr (!HALF) {
            return make_uint4(E::pack(fst[0].x, snd[0].x), E::pack(fst[0].y, snd[0].y),
                              E::pack(fst[1].x, snd[1].x), E::pack(fst[1].y, snd[1].y));
        } else {
            return make_uint4(E::pack(fst[0].x, fst[0].y), E::pack(fst[1].x, fst[1].y),
                              E::pack(snd[0].x, snd[0].y), E::pack(snd[1].x, snd[1].y));
        }
    }

    // Column (element index in the row) of fst[h] (second = false) or snd[h], component k.
    static __device__ __forceinline__ constexpr int col(int sub, int h, bool second, int k)
    {
        return HALF ? (second ? D / 2 : 0) + 4 * sub + 2 * h + k
                    : 8 * sub + 4 * h + 2 * k + (second ? 1 : 0);
    }

    // The lane's weights in the same arrangement (w: d fp32 values, 16-byte aligned).
    static __device__ __forceinline__ void weights(const float* w, int sub, float2 fst[2],
                                                   float2 snd[2])
    {
        if constexpr (!HALF) {
            const float4 a0 = *reinterpret_cast<const float4*>(w + 8 * sub);
            const float4 a1 = *reinterpret_cast<const float4*>(w + 8 * sub + 4);
            fst[0] = make_float2(a0.x, a0.z);
            snd[0] = make_float2(a0.y, a0.w);
            fst[1] = make_float2(a1.x, a1.z);
            snd[1] = make_float2(a1.y, a1.w);
        } else {
            const float4 f = *reinterpret_cast<const float4*>(w + 4 * sub);
            const float4 s = *reinterpret_cast<const float4*>(w + D / 2 + 4 * sub);
            fst[0] = make_float2(f.x, f.y);
            fst[1] = make_float2(f.z, f.w);
            snd[0] = make_float2(s.x, s.y);
            snd[1] = make_float2(s.z, s.w);
        }
    }
};

}  // namespace uly
