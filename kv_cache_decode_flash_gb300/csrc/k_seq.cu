// k_seq.cu - kernels of the sequence operations.
//
// The cold store is built from llama.cpp-style sequence ops ("Plan: lossless
// long context - derived hot/cold sizing + host-RAM KV cold store", section
// llama - KV-byte offload: MemorySeqCopy / MemorySeqRemove / MemorySeqAdd,
// StateSeqGetData / StateSeqSetData).  On the device they reduce to two
// kernels:
//  - copy_runs: runs of consecutive rows of one KV head, copied for every
//    layer and every stored tensor with 16-byte vector moves where
//    alignment allows (seq_cp, compaction in seq_rm, state pack and unpack);
//  - rope_shift: re-rotate stored K head-rows by a position delta (section
//    OpenVINO - KV-byte offload: shifted imports rotate RoPE-positioned keys
//    by the destination/source position delta), dequantising and
//    requantising q8_0 rows in one pass.
#include "kvc_internal.h"

#include <cuda_fp16.h>

namespace kvc {
namespace {

// Copy `bytes` (a multiple of sizeof(T)) with the CTA's threads; each
// thread has U loads in flight before its stores.
__device__ __forceinline__ uint4 flip_bits(uint4 v, uint32_t m) { return make_uint4(v.x ^ m, v.y ^ m, v.z ^ m, v.w ^ m); }
__device__ __forceinline__ uint2 flip_bits(uint2 v, uint32_t m) { return make_uint2(v.x ^ m, v.y ^ m); }
__device__ __forceinline__ uint32_t flip_bits(uint32_t v, uint32_t m) { return v ^ m; }
__device__ __forceinline__ uint8_t flip_bits(uint8_t v, uint32_t m) { return (uint8_t)(v ^ (m & 255u)); }

template <typename T, int U>
__device__ __forceinline__ void copy_vec(const uint8_t *src, uint8_t *dst, int64_t bytes, uint32_t flip = 0) {
    const T *s = reinterpret_cast<const T *>(src);
    T *d = reinterpret_cast<T *>(dst);
    const int64_t n = bytes / (int64_t)sizeof(T);
    const int64_t step = (int64_t)blockDim.x * U;
    for (int64_t i0 = threadIdx.x; i0 < n; i0 += step) {
        T v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (i0 + u * blockDim.x < n) v[u] = flip_bits(s[i0 + u * blockDim.x], flip);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (i0 + u * blockDim.x < n) d[i0 + u * blockDim.x] = v[u];
    }
}

// One CTA per (run, layer, tensor).
__global__ void __launch_bounds__(256) copy_runs_kernel(const __grid_constant__ RunCopyArgs a,
                                                        const RowRun *runs) {
    const int t = blockIdx.z;
    if (!a.base[t]) return;
    const RowRun rn = runs[blockIdx.x];
    const int64_t l = a.l0 + (int64_t)blockIdx.y;
    const int64_t rb = a.rowb[t];
    const int64_t other_rows = a.payload ? a.payload_rows : a.pool_rows;
    if (rn.n < 0 || rn.row0 < 0 || rn.row0 + rn.n > a.pool_rows || rn.other < 0 || rn.other + rn.n > other_rows) {
        if (threadIdx.x == 0 && a.err) atomicOr(a.err, ERR_BAD_INDEX);
        return;
    }
    uint8_t *pool = a.base[t] + (rn.row0 + l * a.pool_rows) * rb;
    uint8_t *other = a.payload ? a.payload + l * a.layer_bytes + a.toff[t] + rn.other * rb
                               : a.base[t] + (rn.other + l * a.pool_rows) * rb;
    const uint8_t *src = (a.payload && !a.to_payload) ? other : pool;
    uint8_t *dst = (a.payload && !a.to_payload) ? pool : other;
    const int64_t bytes = (int64_t)rn.n * rb;
    const uintptr_t al = (uintptr_t)src | (uintptr_t)dst | (uintptr_t)bytes;
    const uint32_t flip = a.flip[t];
    if ((al & 15) == 0)
        copy_vec<uint4, 4>(src, dst, bytes, flip);
    else if ((al & 7) == 0)
        copy_vec<uint2, 4>(src, dst, bytes, flip);
    else if ((al & 3) == 0)
        copy_vec<uint32_t, 4>(src, dst, bytes, flip);
    else
        copy_vec<uint8_t, 4>(src, dst, bytes, flip);
}

struct RopeArgs {
    int mode, n_layer;
    void *kdata;
    uint16_t *kscales;
    int64_t layer_rows;
    const RopeSpan *spans;
    uint32_t *err; // a span outside the layer pool is reported and skipped
    float2 cs[64]; // (cos, sin) of delta * theta_i, i < D/2
};

// Code i of 16 stored offset-binary bytes, as an exact float: the byte goes
// into the low mantissa bits of 2^23 (0x4B0000uu = 2^23 + u), and 2^23 + 128
// is subtracted.
__device__ __forceinline__ float code_at(const uint4 &w, int i) {
    const uint32_t u = i < 4 ? w.x : i < 8 ? w.y : i < 12 ? w.z : w.w;
    uint32_t f;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(f) : "r"(u), "r"(0x4B000000u), "r"(0x7440u | (uint32_t)(i & 3)));
    return __fsub_rn(__uint_as_float(f), 8388736.0f);
}
// 16 rounded codes (integral floats in [-127, 127]) -> 16 offset-binary bytes:
// c + 2^23 + 128 is exact and its low byte is c + 128; PRMTs gather the bytes.
__device__ __forceinline__ uint4 pack16(const float (&c)[16]) {
    uint32_t b[16], u[4];
#pragma unroll
    for (int i = 0; i < 16; ++i) b[i] = __float_as_uint(__fadd_rn(c[i], 8388736.0f));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t lo, hi;
        asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(lo) : "r"(b[4 * j]), "r"(b[4 * j + 1]));
        asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(hi) : "r"(b[4 * j + 2]), "r"(b[4 * j + 3]));
        asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(u[j]) : "r"(lo), "r"(hi));
    }
    return make_uint4(u[0], u[1], u[2], u[3]);
}

// One CTA per (span, layer); TPR threads per head-row, each holding two
// 16-byte pieces A and B of the row:
//   NEOX: A = dims [V k, V k + V), B = A + D/2 (the rotation partners);
//   NORM: A, B = dims [2V k, 2V k + V), [2V k + V, 2V k + 2V) (pairs inside).
// V = 16 values per piece for q8_0 codes, 8 for f16.  A q8_0 block of 32
// dims is the A (or B) pieces of threads k and k ^ 1 (NEOX) or A and B of
// one thread (NORM), so the requantisation max needs at most one shuffle.
// Every thread runs the same number of passes (rows past the span end are
// masked), so the shuffles always see the whole warp.
template <bool Q8, int D, int MODE>
__global__ void __launch_bounds__(256, 4) rope_shift_kernel(const __grid_constant__ RopeArgs a) {
    constexpr int V = Q8 ? 16 : 8;
    constexpr int TPR = D / (2 * V);
    constexpr int RPP = 256 / TPR; // rows per pass of the CTA
    constexpr int NB = D / QK;
    constexpr int HALF = D / 2;
    const RopeSpan sp = a.spans[blockIdx.x];
    if (sp.n < 0 || sp.row0 < 0 || sp.row0 + sp.n > a.layer_rows) { // the whole CTA leaves
        if (threadIdx.x == 0 && a.err) atomicOr(a.err, ERR_BAD_INDEX);
        return;
    }
    const int64_t base = sp.row0 + (int64_t)blockIdx.y * a.layer_rows;
    const int k = threadIdx.x % TPR;
    const int da = MODE == KVC_ROPE_NEOX ? V * k : 2 * V * k; // first dim of A
    const int db = MODE == KVC_ROPE_NEOX ? da + HALF : da + V; // first dim of B
    for (int r0 = 0; r0 < sp.n; r0 += RPP) {
        const int r = r0 + (int)threadIdx.x / TPR;
        const bool live = r < sp.n;
        const int64_t R = base + (live ? r : 0);
        uint4 wa = make_uint4(0, 0, 0, 0), wb = wa;
        float sa = 0.f, sb = 0.f;
        if (live) {
            if constexpr (Q8) {
                const uint8_t *row = reinterpret_cast<const uint8_t *>(a.kdata) + R * D;
                wa = *reinterpret_cast<const uint4 *>(row + da);
                wb = *reinterpret_cast<const uint4 *>(row + db);
                sa = __half2float(__ushort_as_half(a.kscales[R * NB + da / QK]));
                sb = __half2float(__ushort_as_half(a.kscales[R * NB + db / QK]));
            } else {
                const __half *row = reinterpret_cast<const __half *>(a.kdata) + R * D;
                wa = *reinterpret_cast<const uint4 *>(row + da);
                wb = *reinterpret_cast<const uint4 *>(row + db);
            }
        }
        auto xa = [&](int i) {
            if constexpr (Q8) return sa * code_at(wa, i); // exact
            else return __half2float(reinterpret_cast<const __half *>(&wa)[i]);
        };
        auto xb = [&](int i) {
            if constexpr (Q8) return sb * code_at(wb, i);
            else return __half2float(reinterpret_cast<const __half *>(&wb)[i]);
        };
        float ya[V], yb[V];
        if constexpr (MODE == KVC_ROPE_NEOX) {
            // (a, b) = (x_i, x_{i + D/2}) -> (a cos - b sin, a sin + b cos)
#pragma unroll
            for (int i = 0; i < V; ++i) {
                const float c = a.cs[da + i].x, s = a.cs[da + i].y, u = xa(i), v = xb(i);
                ya[i] = __fmaf_rn(u, c, __fmul_rn(-v, s));
                yb[i] = __fmaf_rn(u, s, __fmul_rn(v, c));
            }
        } else {
            // (a, b) = (x_2i, x_2i+1), inside each piece
#pragma unroll
            for (int i = 0; i < V; i += 2) {
                const float2 ta = a.cs[(da + i) / 2], tb = a.cs[(db + i) / 2];
                const float u0 = xa(i), u1 = xa(i + 1), v0 = xb(i), v1 = xb(i + 1);
                ya[i] = __fmaf_rn(u0, ta.x, __fmul_rn(-u1, ta.y));
                ya[i + 1] = __fmaf_rn(u0, ta.y, __fmul_rn(u1, ta.x));
                yb[i] = __fmaf_rn(v0, tb.x, __fmul_rn(-v1, tb.y));
                yb[i + 1] = __fmaf_rn(v0, tb.y, __fmul_rn(v1, tb.x));
            }
        }
        if constexpr (Q8) {
            float ma = 0.f, mb = 0.f;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                ma = fmaxf(ma, fabsf(ya[i]));
                mb = fmaxf(mb, fabsf(yb[i]));
            }
            if constexpr (MODE == KVC_ROPE_NEOX) {
                // the other half of each block sits in thread k ^ 1 of this row
                ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
                mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
            } else {
                ma = mb = fmaxf(ma, mb); // A and B are one block
            }
            const float dA = __fdiv_rn(ma, 127.0f), dB = __fdiv_rn(mb, 127.0f);
            const float iA = (dA != 0.0f) ? __fdiv_rn(1.0f, dA) : 0.0f;
            const float iB = (dB != 0.0f) ? __fdiv_rn(1.0f, dB) : 0.0f;
            if (live) {
                float qa[16], qb[16];
#pragma unroll
                for (int i = 0; i < V; ++i) {
                    qa[i] = roundf(__fmul_rn(ya[i], iA));
                    qb[i] = roundf(__fmul_rn(yb[i], iB));
                }
                uint8_t *row = reinterpret_cast<uint8_t *>(a.kdata) + R * D;
                *reinterpret_cast<uint4 *>(row + da) = pack16(qa);
                *reinterpret_cast<uint4 *>(row + db) = pack16(qb);
                if (MODE != KVC_ROPE_NEOX || (k & 1) == 0) {
                    a.kscales[R * NB + da / QK] = __half_as_ushort(__float2half_rn(dA));
                    if (MODE == KVC_ROPE_NEOX) a.kscales[R * NB + db / QK] = __half_as_ushort(__float2half_rn(dB));
                }
            }
        } else if (live) {
            __half *row = reinterpret_cast<__half *>(a.kdata) + R * D;
            uint4 oa, ob;
            __half *ha = reinterpret_cast<__half *>(&oa), *hb = reinterpret_cast<__half *>(&ob);
#pragma unroll
            for (int i = 0; i < V; ++i) {
                ha[i] = __float2half_rn(ya[i]);
                hb[i] = __float2half_rn(yb[i]);
            }
            *reinterpret_cast<uint4 *>(row + da) = oa;
            *reinterpret_cast<uint4 *>(row + db) = ob;
        }
    }
}

} // namespace

cudaError_t launch_copy_runs(const RunCopyArgs &a, const RowRun *runs_dev, int64_t n_runs, int n_layers,
                             cudaStream_t st) {
    if (n_runs <= 0 || n_layers <= 0) return cudaSuccess;
    if (n_runs > 0x7fffffff || n_layers > 65535) return cudaErrorInvalidValue;
    copy_runs_kernel<<<dim3((unsigned)n_runs, (unsigned)n_layers, 4), 256, 0, st>>>(a, runs_dev);
    return cudaGetLastError();
}

cudaError_t launch_rope_shift(int type_k, int D, int mode, void *kdata, uint16_t *kscales, int64_t layer_rows,
                              int n_layer, const RopeSpan *spans_dev, int64_t n_spans, const float2 *cs,
                              uint32_t *err, cudaStream_t st) {
    if (n_spans <= 0 || n_layer <= 0) return cudaSuccess;
    if (n_spans > 0x7fffffff || n_layer > 65535) return cudaErrorInvalidValue;
    if ((uintptr_t)kdata & 15) return cudaErrorMisalignedAddress; // 16-byte row pieces
    RopeArgs a;
    a.mode = mode;
    a.n_layer = n_layer;
    a.kdata = kdata;
    a.kscales = kscales;
    a.layer_rows = layer_rows;
    a.spans = spans_dev;
    a.err = err;
    for (int i = 0; i < 64; ++i) a.cs[i] = i < D / 2 ? cs[i] : make_float2(1.f, 0.f);
    const dim3 grid((unsigned)n_spans, (unsigned)n_layer);
    const bool q8 = type_k == KVC_Q8_0, neox = mode == KVC_ROPE_NEOX;
#define KVC_ROPE_LAUNCH(Q, DD, M) rope_shift_kernel<Q, DD, M><<<grid, 256, 0, st>>>(a)
    if (D == 128) {
        if (q8)
            neox ? KVC_ROPE_LAUNCH(true, 128, KVC_ROPE_NEOX) : KVC_ROPE_LAUNCH(true, 128, KVC_ROPE_NORM);
        else
            neox ? KVC_ROPE_LAUNCH(false, 128, KVC_ROPE_NEOX) : KVC_ROPE_LAUNCH(false, 128, KVC_ROPE_NORM);
    } else if (D == 64) {
        if (q8)
            neox ? KVC_ROPE_LAUNCH(true, 64, KVC_ROPE_NEOX) : KVC_ROPE_LAUNCH(true, 64, KVC_ROPE_NORM);
        else
            neox ? KVC_ROPE_LAUNCH(false, 64, KVC_ROPE_NEOX) : KVC_ROPE_LAUNCH(false, 64, KVC_ROPE_NORM);
    } else {
        return cudaErrorInvalidValue;
    }
#undef KVC_ROPE_LAUNCH
    return cudaGetLastError();
}

} // namespace kvc
