// k_seq.cu - kernels of the sequence operations.
//
// The cold store is built from llama.cpp-style sequence ops ("Plan: lossless
// long context - derived hot/cold sizing + host-RAM KV cold store", section
// llama - KV-byte offload: MemorySeqCopy / MemorySeqRemove / MemorySeqAdd,
// StateSeqGetData / StateSeqSetData).  On the device they reduce to two
// kernels:
//  - copy_segments: a list of byte ranges copied with 16-byte vector moves
//    where alignment allows (seq_cp, compaction in seq_rm, state pack and
//    unpack);
//  - rope_shift: re-rotate stored K head-rows by a position delta (section
//    OpenVINO - KV-byte offload: shifted imports rotate RoPE-positioned keys
//    by the destination/source position delta), dequantising and
//    requantising q8_0 rows in one pass.
#include "kvc_internal.h"

#include <cuda_fp16.h>

namespace kvc {
namespace {

template <typename T>
__device__ __forceinline__ void copy_vec(const uint8_t *src, uint8_t *dst, int64_t bytes) {
    const T *s = reinterpret_cast<const T *>(src);
    T *d = reinterpret_cast<T *>(dst);
    const int64_t n = bytes / (int64_t)sizeof(T);
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) d[i] = s[i];
}

__global__ void __launch_bounds__(256) copy_segments_kernel(const Segment *segs, int n) {
    for (int i = blockIdx.x; i < n; i += gridDim.x) {
        const Segment sg = segs[i];
        const uintptr_t a = (uintptr_t)sg.src | (uintptr_t)sg.dst | (uintptr_t)sg.bytes;
        if ((a & 15) == 0)
            copy_vec<uint4>(sg.src, sg.dst, sg.bytes);
        else if ((a & 7) == 0)
            copy_vec<uint2>(sg.src, sg.dst, sg.bytes);
        else if ((a & 3) == 0)
            copy_vec<uint32_t>(sg.src, sg.dst, sg.bytes);
        else
            copy_vec<uint8_t>(sg.src, sg.dst, sg.bytes);
    }
}

struct RopeArgs {
    int type_k, mode, n_layer;
    void *kdata;
    uint16_t *kscales;
    int64_t layer_rows;
    const int64_t *rows;
    int64_t n_rows;
    float2 cs[64]; // (cos, sin) of delta * theta_i, i < D/2
};

// One warp per (layer, head-row).  Lane holds EPL consecutive values.
template <int D>
__global__ void __launch_bounds__(256) rope_shift_kernel(const __grid_constant__ RopeArgs a) {
    constexpr int EPL = D / 32, LPB = QK / EPL, HALF = D / 2;
    const int lane = threadIdx.x & 31;
    const int64_t w = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (w >= a.n_rows * a.n_layer) return;
    const int64_t l = w / a.n_rows;
    const int64_t R = a.rows[w % a.n_rows] + l * a.layer_rows;
    float x[EPL];
    if (a.type_k == KVC_Q8_0) {
        const int8_t *row = reinterpret_cast<const int8_t *>(a.kdata) + R * D;
        const float d = __half2float(__ushort_as_half(a.kscales[R * (D / QK) + lane / LPB]));
#pragma unroll
        for (int i = 0; i < EPL; ++i) x[i] = d * (float)row[lane * EPL + i]; // exact
    } else {
        const __half *row = reinterpret_cast<const __half *>(a.kdata) + R * D;
#pragma unroll
        for (int i = 0; i < EPL; ++i) x[i] = __half2float(row[lane * EPL + i]);
    }
    float y[EPL];
    if (a.mode == KVC_ROPE_NEOX) {
        // pair (i, i + D/2): the partner value sits in lane ^ 16 at the same slot
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const float other = __shfl_xor_sync(0xffffffffu, x[e], 16);
            const int dim = lane * EPL + e;
            const int i = dim % HALF;
            const float c = a.cs[i].x, s = a.cs[i].y;
            if (dim < HALF)
                y[e] = __fmaf_rn(x[e], c, __fmul_rn(-other, s)); // a cos - b sin
            else
                y[e] = __fmaf_rn(other, s, __fmul_rn(x[e], c)); // a sin + b cos
        }
    } else {
        // pair (2i, 2i + 1) sits inside the lane
#pragma unroll
        for (int e = 0; e < EPL; e += 2) {
            const int i = (lane * EPL + e) / 2;
            const float c = a.cs[i].x, s = a.cs[i].y;
            y[e] = __fmaf_rn(x[e], c, __fmul_rn(-x[e + 1], s));
            y[e + 1] = __fmaf_rn(x[e], s, __fmul_rn(x[e + 1], c));
        }
    }
    if (a.type_k == KVC_Q8_0) {
        float am = 0.0f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) am = fmaxf(am, fabsf(y[i]));
#pragma unroll
        for (int m = 1; m < LPB; m <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, m));
        const float d = __fdiv_rn(am, 127.0f);
        const float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
        int8_t *row = reinterpret_cast<int8_t *>(a.kdata) + R * D;
#pragma unroll
        for (int i = 0; i < EPL; ++i) row[lane * EPL + i] = (int8_t)(int)roundf(__fmul_rn(y[i], id));
        if ((lane % LPB) == 0) a.kscales[R * (D / QK) + lane / LPB] = __half_as_ushort(__float2half_rn(d));
    } else {
        __half *row = reinterpret_cast<__half *>(a.kdata) + R * D;
#pragma unroll
        for (int i = 0; i < EPL; ++i) row[lane * EPL + i] = __float2half_rn(y[i]);
    }
}

} // namespace

cudaError_t launch_copy_segments(const Segment *segs_dev, int n, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = n < sms * 8 ? n : sms * 8;
    copy_segments_kernel<<<grid, 256, 0, st>>>(segs_dev, n);
    return cudaGetLastError();
}

cudaError_t launch_rope_shift(int type_k, int D, int mode, void *kdata, uint16_t *kscales, int64_t layer_rows,
                              int n_layer, const int64_t *rows_dev, int64_t n_rows, const float2 *cs,
                              cudaStream_t st) {
    if (n_rows <= 0) return cudaSuccess;
    RopeArgs a;
    a.type_k = type_k;
    a.mode = mode;
    a.n_layer = n_layer;
    a.kdata = kdata;
    a.kscales = kscales;
    a.layer_rows = layer_rows;
    a.rows = rows_dev;
    a.n_rows = n_rows;
    for (int i = 0; i < D / 2 && i < 64; ++i) a.cs[i] = cs[i];
    const int64_t warps = n_rows * n_layer;
    const unsigned grid = (unsigned)((warps + 7) / 8);
    if (D == 128)
        rope_shift_kernel<128><<<grid, 256, 0, st>>>(a);
    else if (D == 64)
        rope_shift_kernel<64><<<grid, 256, 0, st>>>(a);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

} // namespace kvc
