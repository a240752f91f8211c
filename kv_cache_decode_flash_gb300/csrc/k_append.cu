// k_append.cu - quantise-on-append and page-table update kernels.
//
// Quantise-on-append writes a token's K and V head-rows into cache cells as
// the model produces them (the per-layer cpy_k/cpy_v set_rows of
// "F5 - Advanced KV Cache Techniques", section M2 - HeadInfer).  q8_0 blocks
// of 32 values get d = max|x| / 127 (IEEE fp32 division), codes
// round-half-away(x * (1/d)) and the scale stored as fp16(d), rounded to
// nearest even; f16 stores fp16(x).  The fp32 step order is fixed, so the
// codes are bit-exact with any implementation of the same steps.
#include "quant_row.cuh"

namespace kvc {
namespace {

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
        store_row<D>(a.type_k, a.dst[i].lv.k, R, lane, xk);
        store_row<D>(a.type_v, a.dst[i].lv.v, R, lane, xv);
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
