// k_keydiff.cu - KeyDiff distinctiveness of a sequence's keys in one layer.
//
// "F5 - Advanced KV Cache Techniques", section M1 (retention-aware context
// shift) evicts the keys that are least distinctive by cosine similarity:
// a row's score is the mean over the KV heads of 1 - cos(key, the head's
// mean key), higher meaning keep.  Two passes over the stored K (post-RoPE;
// q8_0 dequantised exactly):
//  1. keydiff_sum: one CTA per row span (a page run of one KV head) sums its
//     rows' keys; keydiff_mean adds the spans of every head in span order
//     (deterministic) and divides by the row count;
//  2. keydiff_score: one warp per row in position order; each lane takes
//     one 32-element block of one head (a pass covers 32 / NB heads), the
//     dot product with the head's mean and the squared norm are summed over
//     the NB lanes of a head, and the per-head terms over the warp.
#include "kvc_internal.h"

#include <cuda_fp16.h>

namespace kvc {
namespace {

// Four stored values of a row as floats: q8_0 codes (offset binary) times
// the block scale, or f16 halves.
__device__ __forceinline__ void load4(const KeyDiffArgs &a, int64_t R, int d, float (&x)[4]) {
    if (a.q8) {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(a.kdata + R * a.D + d);
        const float s = __half2float(__ushort_as_half(a.kscales[R * (a.D / QK) + d / QK]));
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = s * (float)((int)((w >> (8 * i)) & 255u) - 128); // exact
    } else {
        const uint2 w = *reinterpret_cast<const uint2 *>(a.kdata + (R * a.D + d) * 2);
        const float2 lo = __half22float2(*reinterpret_cast<const __half2 *>(&w.x));
        const float2 hi = __half22float2(*reinterpret_cast<const __half2 *>(&w.y));
        x[0] = lo.x;
        x[1] = lo.y;
        x[2] = hi.x;
        x[3] = hi.y;
    }
}

// Pass 1a: per span, the sum of its rows' keys (head of the span).  128
// threads: D / 4 lanes per row, 128 / (D / 4) rows at a time.
__global__ void __launch_bounds__(128) keydiff_sum_kernel(const __grid_constant__ KeyDiffArgs a) {
    __shared__ float part[128 * 4];
    const RopeSpan sp = a.spans[blockIdx.x];
    const int lanes = a.D / 4, rows_at_once = 128 / lanes;
    const int l = threadIdx.x % lanes, r = threadIdx.x / lanes;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j = r; j < sp.n; j += rows_at_once) {
        float x[4];
        load4(a, sp.row0 + a.layer_off + j, 4 * l, x);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] += x[i];
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) part[threadIdx.x * 4 + i] = acc[i];
    __syncthreads();
    // fixed-order sum over the row groups
    if (threadIdx.x < lanes) {
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        for (int q = 0; q < rows_at_once; ++q)
#pragma unroll
            for (int i = 0; i < 4; ++i) s[i] += part[(q * lanes + threadIdx.x) * 4 + i];
#pragma unroll
        for (int i = 0; i < 4; ++i) a.span_sum[(int64_t)blockIdx.x * a.D + 4 * threadIdx.x + i] = s[i];
    }
}

// Pass 1b: per head, the span sums in span order over the row count; also
// the mean's norm.  One CTA per head, D threads.
__global__ void __launch_bounds__(128) keydiff_mean_kernel(const __grid_constant__ KeyDiffArgs a) {
    const int g = blockIdx.x, d = threadIdx.x;
    __shared__ float sq[128];
    float s = 0.f;
    if (d < a.D) {
        for (int i = 0; i < a.n_spans; ++i)
            if (a.span_head[i] == g) s += a.span_sum[(int64_t)i * a.D + d];
        s /= (float)a.n_rows;
        a.mean[g * a.D + d] = s;
    }
    sq[d] = d < a.D ? s * s : 0.f;
    __syncthreads();
    if (d == 0) {
        float t = 0.f;
        for (int i = 0; i < a.D; ++i) t += sq[i];
        a.mean_norm[g] = sqrtf(t);
    }
}

// Pass 2: one warp per row (position order).  Lane = (head, block) within a
// pass of 32 / NB heads.
__global__ void __launch_bounds__(256) keydiff_score_kernel(const __grid_constant__ KeyDiffArgs a) {
    extern __shared__ float smean[]; // [Hk][D] then [Hk] norms
    for (int i = threadIdx.x; i < a.Hk * a.D; i += blockDim.x) smean[i] = a.mean[i];
    for (int i = threadIdx.x; i < a.Hk; i += blockDim.x) smean[a.Hk * a.D + i] = a.mean_norm[i];
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t j = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (j >= a.n_rows) return; // whole warps leave together
    const int NB = a.D / QK;
    const int heads_per_pass = 32 / NB;
    const int64_t R0 = a.row_base[j] + a.layer_off; // head 0's row; head g's is R0 + g * P
    float score = 0.f;
    for (int g0 = 0; g0 < a.Hk; g0 += heads_per_pass) {
        const int g = g0 + lane / NB, b = lane % NB;
        float dot = 0.f, nn = 0.f;
        if (g < a.Hk) {
            const int64_t R = R0 + (int64_t)g * a.P;
            const float *mu = smean + g * a.D + b * QK;
#pragma unroll 4
            for (int e = 0; e < QK; e += 4) {
                float x[4];
                load4(a, R, b * QK + e, x);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    dot = fmaf(x[i], mu[e + i], dot);
                    nn = fmaf(x[i], x[i], nn);
                }
            }
        }
        // sum over the NB lanes of one head (NB is a power of two dividing 32)
        for (int m = 1; m < NB; m <<= 1) {
            dot += __shfl_xor_sync(0xffffffffu, dot, m);
            nn += __shfl_xor_sync(0xffffffffu, nn, m);
        }
        if (b == 0 && g < a.Hk) {
            const float mn = smean[a.Hk * a.D + g];
            const float c = (nn > 0.f && mn > 0.f) ? dot / (sqrtf(nn) * mn) : 0.f; // degenerate: 0
            score += 1.f - c;
        }
    }
    for (int m = 16; m > 0; m >>= 1) score += __shfl_xor_sync(0xffffffffu, score, m);
    if (lane == 0) a.score[j] = score / (float)a.Hk;
}

} // namespace

cudaError_t launch_keydiff(const KeyDiffArgs &a, cudaStream_t st) {
    if (a.n_rows <= 0) return cudaSuccess;
    if (a.D != 64 && a.D != 128) return cudaErrorInvalidValue;
    keydiff_sum_kernel<<<(unsigned)a.n_spans, 128, 0, st>>>(a);
    keydiff_mean_kernel<<<(unsigned)a.Hk, 128, 0, st>>>(a);
    const size_t smem = ((size_t)a.Hk * a.D + a.Hk) * sizeof(float);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(keydiff_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    const unsigned blocks = (unsigned)((a.n_rows + 7) / 8);
    keydiff_score_kernel<<<blocks, 256, smem, st>>>(a);
    return cudaGetLastError();
}

} // namespace kvc
