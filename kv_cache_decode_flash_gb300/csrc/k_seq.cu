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
    uint32_t *err;   // a span outside the layer pool is reported and skipped
    float c[64];     // cos(delta * theta_i), i < D/2
    float s[64];     // sin(delta * theta_i)
};

// Two-lane fp32 arithmetic (one instruction for both lanes, each lane rounded
// as the scalar IEEE operation would be).
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// Code byte i of 16 stored offset-binary bytes, placed at bits 8..15 of the
// float 2^23: the result is 2^23 + 256 u (u = code + 128), exact.
__device__ __forceinline__ float code_hi(const uint4 &w, int i) {
    const uint32_t u = i < 4 ? w.x : i < 8 ? w.y : i < 12 ? w.z : w.w;
    uint32_t f;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(f) : "r"(u), "r"(0x4B000000u), "r"(0x7504u | ((uint32_t)(i & 3) << 4)));
    return __uint_as_float(f);
}
// Rounding half away from zero of q (|q| < 2^22) is the truncation of
// q + copysign(0.49999997, q) (the predecessor of 1/2): the sum is exact
// except where q lies within half an ulp below a half-integer, and there it
// rounds to a value that truncates the same way.  This gives the bias.
__device__ __forceinline__ float2 half_away_bias(float2 q) {
    return make_float2(__uint_as_float((__float_as_uint(q.x) & 0x80000000u) | 0x3EFFFFFFu),
                       __uint_as_float((__float_as_uint(q.y) & 0x80000000u) | 0x3EFFFFFFu));
}
// Four signed codes (two's complement in the low bytes) -> one word of
// offset-binary bytes.
__device__ __forceinline__ uint32_t pack4(int c0, int c1, int c2, int c3) {
    uint32_t lo, hi, w;
    asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(lo) : "r"(c0), "r"(c1));
    asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(hi) : "r"(c2), "r"(c3));
    asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(w) : "r"(lo), "r"(hi));
    return w ^ 0x80808080u;
}

// One CTA per (span, layer); TPR threads per head-row, each holding two
// 16-byte pieces A and B of the row:
//   NEOX: A = dims [V k, V k + V), B = A + D/2 (the rotation partners);
//   NORM: A, B = dims [2V k, 2V k + V), [2V k + V, 2V k + 2V) (pairs inside).
// V = 16 values per piece for q8_0 codes, 8 for f16.  Either way thread k
// rotates by the V angles theta_{Vk} .. theta_{Vk+V-1}; their cos, sin and
// -sin sit in shared memory.  A q8_0 block of 32 dims is the A (or B)
// pieces of threads k and k ^ 1 (NEOX) or A and B of one thread (NORM), so
// the requantisation max needs at most one shuffle; under NEOX each of the
// two threads divides for one of the two blocks and they swap results.
// Every thread runs the same number of passes (rows past the span end are
// masked), so the shuffles always see the whole warp.
//
// Values are held as lane pairs for the two-lane arithmetic.  Pair t of a
// piece holds elements (2t, 2t+1) under NEOX; under NORM pair 2j holds the
// even elements (4j, 4j+2) and pair 2j+1 the odd ones (4j+1, 4j+3), so one
// two-lane step rotates the adjacent pairs of angles 2j and 2j+1.
template <int MODE>
__device__ __forceinline__ constexpr int pair_elem(int t, int lane) {
    return MODE == KVC_ROPE_NEOX ? 2 * t + lane : 4 * (t / 2) + (t & 1) + 2 * lane;
}

template <bool Q8, int D, int MODE>
__global__ void __launch_bounds__(256, 4) rope_shift_kernel(const __grid_constant__ RopeArgs a) {
    constexpr int V = Q8 ? 16 : 8;
    constexpr int NP = V / 2;      // lane pairs per piece
    constexpr int TPR = D / (2 * V);
    constexpr int RPP = 256 / TPR; // rows per pass of the CTA
    constexpr int NB = D / QK;
    constexpr int HALF = D / 2;
    constexpr int TS = V + 4;      // padded stride of one thread's angles (no bank conflicts)
    constexpr bool NEOX = MODE == KVC_ROPE_NEOX;
    __shared__ __align__(16) float trig[3][TPR * TS];
    const RopeSpan sp = a.spans[blockIdx.x];
    if (sp.n < 0 || sp.row0 < 0 || sp.row0 + sp.n > a.layer_rows) { // the whole CTA leaves
        if (threadIdx.x == 0 && a.err) atomicOr(a.err, ERR_BAD_INDEX);
        return;
    }
    for (int i = threadIdx.x; i < TPR * V; i += blockDim.x) {
        const int o = (i / V) * TS + i % V;
        trig[0][o] = a.c[i];
        trig[1][o] = a.s[i];
        trig[2][o] = -a.s[i];
    }
    __syncthreads();
    const int64_t base = sp.row0 + (int64_t)blockIdx.y * a.layer_rows;
    const int k = threadIdx.x % TPR;
    const int da = NEOX ? V * k : 2 * V * k; // first dim of A
    const int db = NEOX ? da + HALF : da + V; // first dim of B
    const float *tc = &trig[0][k * TS], *tsn = &trig[1][k * TS], *tns = &trig[2][k * TS];
    // the next pass's row pieces are requested before this pass is computed
    auto fetch = [&](int r0, uint4 &wa, uint4 &wb, uint16_t &ha, uint16_t &hb) {
        const int r = r0 + (int)threadIdx.x / TPR;
        if (r < sp.n) {
            const int64_t R = base + r;
            if constexpr (Q8) {
                const uint8_t *row = reinterpret_cast<const uint8_t *>(a.kdata) + R * D;
                wa = *reinterpret_cast<const uint4 *>(row + da);
                wb = *reinterpret_cast<const uint4 *>(row + db);
                ha = a.kscales[R * NB + da / QK];
                hb = a.kscales[R * NB + db / QK];
            } else {
                const __half *row = reinterpret_cast<const __half *>(a.kdata) + R * D;
                wa = *reinterpret_cast<const uint4 *>(row + da);
                wb = *reinterpret_cast<const uint4 *>(row + db);
            }
        }
    };
    uint4 wa = make_uint4(0, 0, 0, 0), wb = wa;
    uint16_t ha = 0, hb = 0;
    fetch(0, wa, wb, ha, hb);
    for (int r0 = 0; r0 < sp.n; r0 += RPP) {
        const int r = r0 + (int)threadIdx.x / TPR;
        const bool live = r < sp.n;
        const int64_t R = base + (live ? r : 0);
        uint4 nwa = make_uint4(0, 0, 0, 0), nwb = nwa;
        uint16_t nha = 0, nhb = 0;
        if (r0 + RPP < sp.n) fetch(r0 + RPP, nwa, nwb, nha, nhb);
        const float sa = __half2float(__ushort_as_half(ha)), sb = __half2float(__ushort_as_half(hb));
        // dequantise into lane pairs.  q8_0: x = s (u - 128) as one FMA of
        // 2^23 + 256 u by s/256 minus (2^23 + 2^15) s/256; the constant has
        // 9 significant bits and s 11, so every term is exact.
        float2 xa[NP], xb[NP];
        if constexpr (Q8) {
            const float sa8 = sa * (1.0f / 256.0f), sb8 = sb * (1.0f / 256.0f);
            const float2 ma2 = make_float2(sa8, sa8), mb2 = make_float2(sb8, sb8);
            const float oa = -8421376.0f * sa8, ob = -8421376.0f * sb8;
            const float2 oa2 = make_float2(oa, oa), ob2 = make_float2(ob, ob);
#pragma unroll
            for (int t = 0; t < NP; ++t) {
                const int e0 = pair_elem<MODE>(t, 0), e1 = pair_elem<MODE>(t, 1);
                xa[t] = fma2(make_float2(code_hi(wa, e0), code_hi(wa, e1)), ma2, oa2);
                xb[t] = fma2(make_float2(code_hi(wb, e0), code_hi(wb, e1)), mb2, ob2);
            }
        } else {
            const __half *ha = reinterpret_cast<const __half *>(&wa), *hb = reinterpret_cast<const __half *>(&wb);
#pragma unroll
            for (int t = 0; t < NP; ++t) {
                const int e0 = pair_elem<MODE>(t, 0), e1 = pair_elem<MODE>(t, 1);
                xa[t] = make_float2(__half2float(ha[e0]), __half2float(ha[e1]));
                xb[t] = make_float2(__half2float(hb[e0]), __half2float(hb[e1]));
            }
        }
        // rotate: (u, v) -> (u cos - v sin, u sin + v cos), the products v sin
        // and v cos rounded before the fused multiply-add
        float2 ya[NP], yb[NP];
#pragma unroll
        for (int m = 0; m < V / 4; ++m) { // angles 4m .. 4m+3 of this thread
            const float4 c4 = *reinterpret_cast<const float4 *>(tc + 4 * m);
            const float4 s4 = *reinterpret_cast<const float4 *>(tsn + 4 * m);
            const float4 n4 = *reinterpret_cast<const float4 *>(tns + 4 * m);
#pragma unroll
            for (int h = 0; h < 2; ++h) { // angle pair 2m + h
                const float2 c2 = h ? make_float2(c4.z, c4.w) : make_float2(c4.x, c4.y);
                const float2 s2 = h ? make_float2(s4.z, s4.w) : make_float2(s4.x, s4.y);
                const float2 n2 = h ? make_float2(n4.z, n4.w) : make_float2(n4.x, n4.y);
                const int j = 2 * m + h;
                if constexpr (NEOX) {
                    ya[j] = fma2(xa[j], c2, mul2(xb[j], n2));
                    yb[j] = fma2(xa[j], s2, mul2(xb[j], c2));
                } else if (j < V / 4) { // piece A: even pair 2j, odd pair 2j+1
                    ya[2 * j] = fma2(xa[2 * j], c2, mul2(xa[2 * j + 1], n2));
                    ya[2 * j + 1] = fma2(xa[2 * j], s2, mul2(xa[2 * j + 1], c2));
                } else { // piece B
                    const int i = j - V / 4;
                    yb[2 * i] = fma2(xb[2 * i], c2, mul2(xb[2 * i + 1], n2));
                    yb[2 * i + 1] = fma2(xb[2 * i], s2, mul2(xb[2 * i + 1], c2));
                }
            }
        }
        if constexpr (Q8) {
            float ma = 0.f, mb = 0.f;
#pragma unroll
            for (int t = 0; t < NP; ++t) {
                ma = fmaxf(ma, fmaxf(fabsf(ya[t].x), fabsf(ya[t].y)));
                mb = fmaxf(mb, fmaxf(fabsf(yb[t].x), fabsf(yb[t].y)));
            }
            float iA, iB, d_own;
            if constexpr (NEOX) {
                // the other half of each block sits in thread k ^ 1 of this row
                ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
                mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
                const bool odd = k & 1; // even: A's block, odd: B's block (scale and reciprocal)
                d_own = __fdiv_rn(odd ? mb : ma, 127.0f);
                const float i_own = (d_own != 0.0f) ? __fdiv_rn(1.0f, d_own) : 0.0f;
                const float i_oth = __shfl_xor_sync(0xffffffffu, i_own, 1);
                iA = odd ? i_oth : i_own;
                iB = odd ? i_own : i_oth;
            } else {
                ma = fmaxf(ma, mb); // A and B are one block
                d_own = __fdiv_rn(ma, 127.0f);
                iA = iB = (d_own != 0.0f) ? __fdiv_rn(1.0f, d_own) : 0.0f;
            }
            if (live) {
                int ca[V], cb[V];
                const float2 ia2 = make_float2(iA, iA), ib2 = make_float2(iB, iB);
#pragma unroll
                for (int t = 0; t < NP; ++t) {
                    const float2 qa = mul2(ya[t], ia2), qb = mul2(yb[t], ib2);
                    const float2 pa = add2(qa, half_away_bias(qa)), pb = add2(qb, half_away_bias(qb));
                    const int e0 = pair_elem<MODE>(t, 0), e1 = pair_elem<MODE>(t, 1);
                    ca[e0] = __float2int_rz(pa.x);
                    ca[e1] = __float2int_rz(pa.y);
                    cb[e0] = __float2int_rz(pb.x);
                    cb[e1] = __float2int_rz(pb.y);
                }
                uint8_t *row = reinterpret_cast<uint8_t *>(a.kdata) + R * D;
                *reinterpret_cast<uint4 *>(row + da) = make_uint4(pack4(ca[0], ca[1], ca[2], ca[3]),
                                                                  pack4(ca[4], ca[5], ca[6], ca[7]),
                                                                  pack4(ca[8], ca[9], ca[10], ca[11]),
                                                                  pack4(ca[12], ca[13], ca[14], ca[15]));
                *reinterpret_cast<uint4 *>(row + db) = make_uint4(pack4(cb[0], cb[1], cb[2], cb[3]),
                                                                  pack4(cb[4], cb[5], cb[6], cb[7]),
                                                                  pack4(cb[8], cb[9], cb[10], cb[11]),
                                                                  pack4(cb[12], cb[13], cb[14], cb[15]));
                if constexpr (NEOX) {
                    a.kscales[R * NB + ((k & 1) ? db : da) / QK] = __half_as_ushort(__float2half_rn(d_own));
                } else {
                    a.kscales[R * NB + da / QK] = __half_as_ushort(__float2half_rn(d_own));
                }
            }
        } else if (live) {
            __half *row = reinterpret_cast<__half *>(a.kdata) + R * D;
            float fa[V], fb[V];
#pragma unroll
            for (int t = 0; t < NP; ++t) {
                fa[pair_elem<MODE>(t, 0)] = ya[t].x;
                fa[pair_elem<MODE>(t, 1)] = ya[t].y;
                fb[pair_elem<MODE>(t, 0)] = yb[t].x;
                fb[pair_elem<MODE>(t, 1)] = yb[t].y;
            }
            uint4 oa, ob;
            __half2 *ha = reinterpret_cast<__half2 *>(&oa), *hb = reinterpret_cast<__half2 *>(&ob);
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                ha[i] = __floats2half2_rn(fa[2 * i], fa[2 * i + 1]);
                hb[i] = __floats2half2_rn(fb[2 * i], fb[2 * i + 1]);
            }
            *reinterpret_cast<uint4 *>(row + da) = oa;
            *reinterpret_cast<uint4 *>(row + db) = ob;
        }
        wa = nwa;
        wb = nwb;
        ha = nha;
        hb = nhb;
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
    for (int i = 0; i < 64; ++i) {
        a.c[i] = i < D / 2 ? cs[i].x : 1.f;
        a.s[i] = i < D / 2 ? cs[i].y : 0.f;
    }
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
