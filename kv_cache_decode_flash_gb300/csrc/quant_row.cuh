// quant_row.cuh - quantise-on-append of one head-row by one warp.
//
// Shared by the append kernel and the attention kernel's fused append (the
// decode step), so that a row stored by either is the same bytes.  q8_0
// blocks of 32 values get d = max|x| / 127 (IEEE fp32 division), codes
// round-half-away(x * (1/d)) and the scale stored as fp16(d), rounded to
// nearest even; f16 stores fp16(x) ("F5 - Advanced KV Cache Techniques",
// section M2 - HeadInfer: the per-layer cpy_k/cpy_v writes; the q8_0 block
// of the decode-attention statement).
#pragma once

#include "kvc_internal.h"

#include <cuda_fp16.h>

namespace kvc {

// Elements per lane for a head-row of D values handled by one warp.
template <int D>
struct RowShape {
    static constexpr int EPL = D / 32;   // 2 (D=64) or 4 (D=128)
    static constexpr int LPB = QK / EPL; // lanes per q8_0 block
};

template <int EPL>
__device__ __forceinline__ void load_row(const float *src, int lane, float (&x)[EPL]) {
    if constexpr (EPL == 4) {
        float4 t = reinterpret_cast<const float4 *>(src)[lane];
        x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
    } else {
        float2 t = reinterpret_cast<const float2 *>(src)[lane];
        x[0] = t.x; x[1] = t.y;
    }
}

// q8_0 of the lane's EPL values within its block of 32 (LPB lanes per block).
template <int EPL, int LPB>
__device__ __forceinline__ void quantise(const float (&x)[EPL], int8_t (&q)[EPL], float &d) {
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) a = fmaxf(a, fabsf(x[i]));
#pragma unroll
    for (int m = 1; m < LPB; m <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
    d = __fdiv_rn(a, 127.0f);
    float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) q[i] = (int8_t)(int)roundf(__fmul_rn(x[i], id));
}

// q4_0 of the lane's EPL values within its block of 32 (LPB lanes per block,
// lane m of a block holding elements m*EPL .. m*EPL + EPL - 1): m = the element
// of largest magnitude, sign kept, the first one on ties; d = m / -8;
// code = min(15, trunc(x * (1/d) + 8.5)), the product and the sum each
// rounded to fp32.
template <int EPL, int LPB>
__device__ __forceinline__ void quantise_q4(const float (&x)[EPL], int lane, int (&c)[EPL], float &d) {
    float a = 0.0f, m = 0.0f;
    int idx = 1 << 30; // no element above magnitude 0: m stays +0
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const float ax = fabsf(x[i]);
        if (ax > a) {
            a = ax;
            m = x[i];
            idx = (lane % LPB) * EPL + i;
        }
    }
#pragma unroll
    for (int o = 1; o < LPB; o <<= 1) {
        const float a2 = __shfl_xor_sync(0xffffffffu, a, o), m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
        if (a2 > a || (a2 == a && i2 < idx)) {
            a = a2;
            m = m2;
            idx = i2;
        }
    }
    d = __fdiv_rn(m, -8.0f);
    const float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) c[i] = min(15, __float2int_rz(__fadd_rn(__fmul_rn(x[i], id), 8.5f)));
}

// Store the warp's head-row x into pool row R of tensor tv (q8_0 codes in
// offset binary, as the attention kernel reads them; q4_0 codes packed, byte
// j of a block holding codes j and j + 16).
template <int D>
__device__ __forceinline__ void store_row(int type, const TensorView &tv, int64_t R, int lane,
                                          const float (&x)[D / 32]) {
    constexpr int EPL = RowShape<D>::EPL, LPB = RowShape<D>::LPB;
    if (type == KVC_Q8_0) {
        int8_t q[EPL];
        float d;
        quantise<EPL, LPB>(x, q, d);
        int8_t *row = reinterpret_cast<int8_t *>(tv.data) + R * D;
        if constexpr (EPL == 4) {
            uint32_t w = (uint32_t)(uint8_t)q[0] | ((uint32_t)(uint8_t)q[1] << 8) |
                         ((uint32_t)(uint8_t)q[2] << 16) | ((uint32_t)(uint8_t)q[3] << 24);
            reinterpret_cast<uint32_t *>(row)[lane] = w ^ CODE_FLIP;
        } else {
            uint16_t w = (uint16_t)((uint16_t)(uint8_t)q[0] | ((uint16_t)(uint8_t)q[1] << 8));
            reinterpret_cast<uint16_t *>(row)[lane] = (uint16_t)(w ^ (CODE_FLIP & 0xffffu));
        }
        if ((lane % LPB) == 0) tv.scales[R * (D / QK) + lane / LPB] = __half_as_ushort(__float2half_rn(d));
    } else if (type == KVC_Q4_0) {
        int c[EPL];
        float d;
        quantise_q4<EPL, LPB>(x, lane, c, d);
        // lane m < LPB/2 holds codes of bytes m*EPL..; its partner m + LPB/2 the codes 16 above
        uint32_t mine = 0;
#pragma unroll
        for (int i = 0; i < EPL; ++i) mine |= (uint32_t)c[i] << (8 * i);
        const uint32_t hi = __shfl_xor_sync(0xffffffffu, mine, LPB / 2);
        const uint32_t w = mine | (hi << 4);
        const int m = lane % LPB;
        if (m < LPB / 2) {
            uint8_t *row = reinterpret_cast<uint8_t *>(tv.data) + R * (D / 2) + (lane / LPB) * (QK / 2) + m * EPL;
            if constexpr (EPL == 4)
                *reinterpret_cast<uint32_t *>(row) = w;
            else
                *reinterpret_cast<uint16_t *>(row) = (uint16_t)w;
        }
        if (m == 0) tv.scales[R * (D / QK) + lane / LPB] = __half_as_ushort(__float2half_rn(d));
    } else {
        __half *row = reinterpret_cast<__half *>(tv.data) + R * D;
#pragma unroll
        for (int i = 0; i < EPL; ++i) row[lane * EPL + i] = __float2half_rn(x[i]);
    }
}

} // namespace kvc
