// k_append.cu - quantise-on-append and page-table update kernels.
//
// Quantise-on-append writes a token's K and V head-rows into cache cells as
// the model produces them (the per-layer cpy_k/cpy_v set_rows of
// "F5 - Advanced KV Cache Techniques", section M2 - HeadInfer).  q8_0 blocks
// of 32 values get d = max|x| / 127 (IEEE fp32 division), codes
// round-half-away(x * (1/d)) and the scale stored as fp16(d), rounded to
// nearest even; f16 stores fp16(x).  The fp32 step order is fixed, so the
// codes are bit-exact with any implementation of the same steps.
#include "kvc_internal.h"

#include <cuda_fp16.h>

namespace kvc {
namespace {

// Elements per lane for a head-row of D values handled by one warp.
template <int D>
struct RowShape {
    static constexpr int EPL = D / 32;          // 2 (D=64) or 4 (D=128)
    static constexpr int LPB = QK / EPL;        // lanes per q8_0 block
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

__device__ __forceinline__ int64_t dst_row(const AppendDst &d, int t, int g, int Hk) {
    int64_t L = (int64_t)d.row0 + t;
    int64_t page, cell;
    if (d.pt) {
        int64_t lr = L + d.off;
        page = d.pt[lr / d.P];
        cell = lr % d.P;
    } else {
        page = 0;
        cell = L;
    }
    return (page * Hk + g) * (int64_t)d.P + cell;
}

template <int D>
__device__ __forceinline__ void store_tensor(int type, const TensorView &tv, int64_t R, int lane,
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
            reinterpret_cast<uint32_t *>(row)[lane] = w ^ CODE_FLIP; // stored offset binary
        } else {
            uint16_t w = (uint16_t)((uint16_t)(uint8_t)q[0] | ((uint16_t)(uint8_t)q[1] << 8));
            reinterpret_cast<uint16_t *>(row)[lane] = (uint16_t)(w ^ (CODE_FLIP & 0xffffu)); // offset binary
        }
        if ((lane % LPB) == 0) tv.scales[R * (D / QK) + lane / LPB] = __half_as_ushort(__float2half_rn(d));
    } else {
        __half *row = reinterpret_cast<__half *>(tv.data) + R * D;
#pragma unroll
        for (int i = 0; i < EPL; ++i) row[lane * EPL + i] = __float2half_rn(x[i]);
    }
}

struct AppendArgs {
    int type_k, type_v, Hk, n_tok, n_dst;
    int in_heads; // head-rows per token in k / v (>= Hk: a context holding a subset of the heads)
    const float *k, *v;
    AppendDst dst[2];
};

// One warp per (token, kv head) head-row.
template <int D>
__global__ void __launch_bounds__(256) append_kernel(const __grid_constant__ AppendArgs a) {
    constexpr int EPL = RowShape<D>::EPL;
    // Let the next kernel (typically this layer's attention) be scheduled now:
    // it only reads rows below the ones written here before its own wait.
    // Inputs may come from the preceding kernel, so wait before reading them.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int64_t w = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (w >= (int64_t)a.n_tok * a.Hk) return;
    const int t = (int)(w / a.Hk), g = (int)(w % a.Hk);
    float xk[EPL], xv[EPL];
    const int64_t in = ((int64_t)t * a.in_heads + g) * D;
    load_row<EPL>(a.k + in, lane, xk);
    load_row<EPL>(a.v + in, lane, xv);
    for (int i = 0; i < a.n_dst; ++i) {
        const int64_t R = dst_row(a.dst[i], t, g, a.Hk);
        store_tensor<D>(a.type_k, a.dst[i].lv.k, R, lane, xk);
        store_tensor<D>(a.type_v, a.dst[i].lv.v, R, lane, xv);
    }
}

struct PtArgs {
    int32_t *pt;
    int n;
    int32_t idx[32];
    int32_t val[32];
};

__global__ void pt_update_kernel(const __grid_constant__ PtArgs a) {
    int i = threadIdx.x;
    if (i < a.n) a.pt[a.idx[i]] = a.val[i];
}

} // namespace

cudaError_t launch_append(int type_k, int type_v, int Hk, int in_heads, int D, int n_tok, const float *k,
                          const float *v, const AppendDst *dst, int n_dst, cudaStream_t st) {
    AppendArgs a;
    a.type_k = type_k;
    a.type_v = type_v;
    a.Hk = Hk;
    a.in_heads = in_heads;
    a.n_tok = n_tok;
    a.n_dst = n_dst;
    a.k = k;
    a.v = v;
    for (int i = 0; i < n_dst && i < 2; ++i) a.dst[i] = dst[i];
    const int64_t warps = (int64_t)n_tok * Hk;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((warps + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (D == 128) return cudaLaunchKernelEx(&cfg, append_kernel<128>, a);
    if (D == 64) return cudaLaunchKernelEx(&cfg, append_kernel<64>, a);
    return cudaErrorInvalidValue;
}

cudaError_t launch_pt_update(int32_t *pt, int n, const int32_t *idx, const int32_t *val, cudaStream_t st) {
    while (n > 0) {
        PtArgs a;
        a.pt = pt;
        a.n = n < 32 ? n : 32;
        for (int i = 0; i < a.n; ++i) {
            a.idx[i] = idx[i];
            a.val[i] = val[i];
        }
        pt_update_kernel<<<1, 32, 0, st>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        idx += a.n;
        val += a.n;
        n -= a.n;
    }
    return cudaSuccess;
}

} // namespace kvc
