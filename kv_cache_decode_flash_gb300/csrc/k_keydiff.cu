// k_keydiff.cu - KeyDiff distinctiveness of a sequence's keys in one layer.
//
// "F5 - Advanced KV Cache Techniques", section M1 (retention-aware context
// shift) evicts the keys that are least distinctive by cosine similarity:
// a row's score is the mean over the KV heads of 1 - cos(key, the head's
// mean key), higher meaning keep.  Two passes over the stored K (post-RoPE;
// q8_0 dequantised exactly).  The sequence's rows come as blocks of at most
// block_rows consecutive rows of one page (head 0's rows; head g's are g * P
// rows further), so a block's rows of one head are one contiguous stretch
// of codes and one of scales, moved into shared memory by bulk async copies:
//  1. keydiff_sum: one CTA per (KV head, slice of KD_WARPS blocks), one warp
//     per block, sums the rows' keys; keydiff_mean adds each head's slices
//     in slice order (deterministic) and divides by the row count;
//  2. keydiff_score: one persistent CTA per SM streams blocks through a
//     KD_STAGES-deep ring (all heads of a block per stage); one lane per
//     (row, head) pair; the per-head terms of a row are added in head order.
// Every wait on a copy is bounded: past the limit the kernel records
// ERR_WAIT_TIMEOUT, waits (bounded) for its copies still in flight and
// stops.
#include "kvc_internal.h"

#include <cuda_fp16.h>

namespace kvc {
namespace {

constexpr int KD_WARPS = 8;        // sum kernel: warps (blocks) per CTA
constexpr int KD_SCORE_WARPS = 8;  // score kernel consumer warps (plus one producer warp)
constexpr int KD_STAGES = 3;       // score kernel ring depth
constexpr int KD_SMEM_MAX = 227 * 1024;
constexpr uint32_t KD_WAIT_LIMIT = 1u << 24;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, unsigned parity) {
    for (uint32_t i = 0; i < KD_WAIT_LIMIT; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
__device__ __forceinline__ void bulk_load(void *dst, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Shared-memory geometry of one head's stretch of a block.
struct Geom {
    int rb;  // row bytes (codes or halves)
    int sb;  // scale bytes per row (q8_0), else 0
    int hsb; // code stretch stride: block_rows * rb, plus 64 bytes for 4-chunk rows when that stride is a
             // multiple of 128 (lanes on eight heads then start on distinct bank groups)
    int srs; // scale stretch stride: the copied 16-byte-aligned superset, block_rows * sb + 16 rounded up
};
__host__ __device__ inline Geom geom(bool q8, int D, int br) {
    Geom g;
    g.rb = q8 ? D : 2 * D;
    g.sb = q8 ? 2 * (D / QK) : 0;
    const int ch = g.rb / 16;
    g.hsb = br * g.rb + ((ch == 4 && (br * ch) % 8 == 0) ? 64 : 0);
    g.srs = q8 ? (br * g.sb + 16 + 15) / 16 * 16 : 0;
    return g;
}
__host__ __device__ inline int score_items(int Hk) {
    return (Hk >= 32 ? 1 : 32 / Hk) * Hk;
}
// Score kernel shared memory: barriers, KD_STAGES stages, padded means,
// norms, per-warp head terms.
// means as padded fp32 rows (f16) or as digit planes (q8_0), norms, fixed-
// point steps (q8_0), per-warp head terms.
__host__ __device__ inline size_t score_mean_bytes(bool q8, int Hk, int D) {
    return q8 ? (size_t)Hk * 3 * D : (size_t)Hk * (D + 4) * 4;
}
__host__ __device__ inline size_t score_smem(bool q8, int Hk, int D, int br) {
    const Geom g = geom(q8, D, br);
    return 128 + (size_t)KD_STAGES * Hk * (g.hsb + g.srs) + score_mean_bytes(q8, Hk, D) + (size_t)Hk * 8 +
           (size_t)KD_SCORE_WARPS * 2 * score_items(Hk) * 4;
}

// One block's stretch of head g: issue its code (and scale) copies on bar.
// Returns the bytes the copies deliver.
__device__ __forceinline__ uint32_t issue_head(const KeyDiffArgs &a, const Geom &G, const KeyDiffBlock &bk, int g,
                                               uint8_t *codes_dst, uint8_t *scales_dst, uint64_t *bar, bool go) {
    const int64_t row = bk.row0 + a.layer_off + (int64_t)g * a.P;
    uint32_t bytes = (uint32_t)(bk.n * G.rb);
    if (go) bulk_load(codes_dst, a.kdata + row * G.rb, (unsigned)(bk.n * G.rb), bar);
    if (G.sb) {
        const uintptr_t s0 = reinterpret_cast<uintptr_t>(a.kscales) + (uintptr_t)(row * G.sb);
        const uintptr_t al = s0 & ~(uintptr_t)15;
        const uint32_t len = (uint32_t)(((s0 - al) + (uintptr_t)(bk.n * G.sb) + 15) / 16 * 16);
        if (go) bulk_load(scales_dst, reinterpret_cast<const void *>(al), len, bar);
        bytes += len;
    }
    return bytes;
}
// Offset of a stretch's first scale inside its 16-byte-aligned copy.
__device__ __forceinline__ int scale_skew(const KeyDiffArgs &a, int64_t row, int sb) {
    return (int)((reinterpret_cast<uintptr_t>(a.kscales) + (uintptr_t)(row * sb)) & 15);
}

// A piece of 16 q8_0 codes (offset binary, code + 128) as exact floats:
// the byte goes under the exponent of 2^23 and 2^23 + 128 is subtracted.
__device__ __forceinline__ float code_at(uint32_t word, int i) {
    return __int_as_float((int)__byte_perm(word, 0x4B000000u, 0x7540u | (unsigned)i)) - 8388736.f;
}

// Pass 1a: CTA (g, c) sums head g's rows of blocks c * KD_WARPS + w, warp
// w taking one block.  Lane 0 of the warp copies the block's stretch into
// the warp's part of shared memory; a lane then adds piece lane % LPR of
// rows lane / LPR, + 32 / LPR, ... (LPR = row bytes / 16).
template <bool Q8, int D>
__global__ void __launch_bounds__(KD_WARPS * 32) keydiff_sum_kernel(const __grid_constant__ KeyDiffArgs a) {
    constexpr int EL = Q8 ? 16 : 8, RB = Q8 ? D : 2 * D, LPR = RB / 16, STEP = 32 / LPR;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t bar[KD_WARPS];
    const Geom G = geom(Q8, D, a.block_rows);
    const int g = blockIdx.x % a.Hk, c = blockIdx.x / a.Hk;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int l = lane % LPR, ro = lane / LPR;
    const int b = c * KD_WARPS + w;
    uint8_t *st = smem + (size_t)w * (G.hsb + G.srs);
    float acc[EL];
#pragma unroll
    for (int i = 0; i < EL; ++i) acc[i] = 0.f;
    if (b < a.n_blocks) {
        const KeyDiffBlock bk = a.blocks[b];
        if (lane == 0) {
            mbar_init(&bar[w], 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            mbar_expect_tx(&bar[w], issue_head(a, G, bk, g, st, st + G.hsb, &bar[w], false));
            issue_head(a, G, bk, g, st, st + G.hsb, &bar[w], true);
        }
        __syncwarp();
        if (mbar_wait_bounded(&bar[w], 0)) {
            const int64_t row = bk.row0 + a.layer_off + (int64_t)g * a.P;
            const uint8_t *sc = st + G.hsb + (Q8 ? scale_skew(a, row, G.sb) : 0);
#pragma unroll 4
            for (int j = ro; j < bk.n; j += STEP) {
                const uint4 v = *reinterpret_cast<const uint4 *>(st + j * RB + 16 * l);
                const uint32_t u[4] = {v.x, v.y, v.z, v.w};
                if constexpr (Q8) {
                    const float s = __half2float(
                        *reinterpret_cast<const __half *>(sc + j * G.sb + 2 * ((EL * l) / QK)));
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[i] = fmaf(code_at(u[i >> 2], i & 3), s, acc[i]);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&u[i]));
                        acc[2 * i] += f.x;
                        acc[2 * i + 1] += f.y;
                    }
                }
            }
        } else {
            if (lane == 0) {
                atomicOr(a.err, ERR_WAIT_TIMEOUT);
                mbar_wait_bounded(&bar[w], 0); // the copies still in flight
            }
            __syncwarp();
        }
    }
    __syncthreads(); // every warp is done with its stretch: reuse the space
    float *part = reinterpret_cast<float *>(smem);
#pragma unroll
    for (int i = 0; i < EL; ++i) part[threadIdx.x * EL + i] = acc[i];
    __syncthreads();
    // fixed-order sum over the CTA's row groups q = w * STEP + ro (thread
    // q * LPR + l holds piece l): thread d < D owns dimension d
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float sum = 0.f;
        for (int q = 0; q < KD_WARPS * STEP; ++q) sum += part[q * D + d];
        a.slice_sum[((int64_t)g * a.n_slices + c) * D + d] = sum;
    }
}

// Pass 1b: per head, the slice sums in slice order over the row count, and
// the mean's norm.  One CTA per head; thread (p, d) adds slices p, p + K,
// ... of dimension d (K = blockDim / D), then the K partials in order.
__global__ void __launch_bounds__(1024) keydiff_mean_kernel(const __grid_constant__ KeyDiffArgs a) {
    __shared__ float part[1024];
    __shared__ float sq[128];
    const int g = blockIdx.x, K = blockDim.x / a.D;
    const int p = threadIdx.x / a.D, d = threadIdx.x % a.D;
    const float *src = a.slice_sum + (int64_t)g * a.n_slices * a.D + d;
    float s = 0.f;
#pragma unroll 8
    for (int c = p; c < a.n_slices; c += K) s += src[(int64_t)c * a.D];
    part[threadIdx.x] = s;
    __syncthreads();
    if (threadIdx.x < a.D) {
        float t = 0.f;
        for (int q = 0; q < K; ++q) t += part[q * a.D + threadIdx.x];
        t /= (float)a.n_rows;
        a.mean[g * a.D + threadIdx.x] = t;
        sq[threadIdx.x] = t * t;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        float t = 0.f;
        for (int i = threadIdx.x; i < a.D; i += 32) t += sq[i];
        for (int m = 16; m > 0; m >>= 1) t += __shfl_xor_sync(0xffffffffu, t, m);
        if (threadIdx.x == 0) a.mean_norm[g] = sqrtf(t);
    }
}

// The dot product of one stored row with the head's mean, and the row's
// squared norm.  The row's 16-byte chunks are taken in a lane-rotated order
// (rot), so the eight lanes of a quarter warp read distinct bank groups.
//
// q8_0: the mean of the head is held as 24-bit fixed point, q = mu / ms
// (ms = max |mu| / QMAX), in three signed base-256 digits (planes hi, mid,
// lo of D int8 each), so a 32-code block's dot product with it is exact
// integer arithmetic: three dp4a per four signed codes, plus one for the
// integer sum of squares.  The block's scale multiplies both once; the
// chunks of one block are visited together (in either order: the integer
// sums do not care).  f16: fp32 products of the halves with the mean.
constexpr int QMAX = 127 * 65536 + 127 * 256 + 127;

template <bool Q8, int D, int NR>
__device__ __forceinline__ void row_terms(const uint8_t *row, int row_stride, const uint8_t *sc, int sc_stride,
                                          const float *mu, const int8_t *digits, int rot, float (&dot)[NR],
                                          float (&nn)[NR]) {
    constexpr int CH = (Q8 ? D : 2 * D) / 16;
#pragma unroll
    for (int r = 0; r < NR; ++r) dot[r] = nn[r] = 0.f;
    if constexpr (Q8) {
        constexpr int NB = D / QK; // scale blocks
#pragma unroll
        for (int kb = 0; kb < NB; ++kb) {
            const int b = (kb + (rot >> 1)) & (NB - 1);
            int dh[NR], dm[NR], dl[NR], inn[NR];
#pragma unroll
            for (int r = 0; r < NR; ++r) dh[r] = dm[r] = dl[r] = inn[r] = 0;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int c = 2 * b + (j ^ (rot & 1));
                const uint4 h = *reinterpret_cast<const uint4 *>(digits + 16 * c);
                const uint4 m = *reinterpret_cast<const uint4 *>(digits + D + 16 * c);
                const uint4 l = *reinterpret_cast<const uint4 *>(digits + 2 * D + 16 * c);
                const uint32_t H[4] = {h.x, h.y, h.z, h.w}, M[4] = {m.x, m.y, m.z, m.w}, L[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(row + r * row_stride + 16 * c);
                    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int wi = 0; wi < 4; ++wi) {
                        const int sw = (int)(u[wi] ^ 0x80808080u); // signed codes
                        inn[r] = __dp4a(sw, sw, inn[r]);
                        dh[r] = __dp4a(sw, (int)H[wi], dh[r]);
                        dm[r] = __dp4a(sw, (int)M[wi], dm[r]);
                        dl[r] = __dp4a(sw, (int)L[wi], dl[r]);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const float t = fmaf((float)dh[r], 65536.f, fmaf((float)dm[r], 256.f, (float)dl[r]));
                const float s = __half2float(*reinterpret_cast<const __half *>(sc + r * sc_stride + 2 * b));
                dot[r] = fmaf(s, t, dot[r]);
                nn[r] = fmaf(s * s, (float)inn[r], nn[r]);
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            const int c = (k + rot) & (CH - 1);
            const float4 m0 = *reinterpret_cast<const float4 *>(mu + 8 * c);
            const float4 m1 = *reinterpret_cast<const float4 *>(mu + 8 * c + 4);
            const float mv[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const uint4 v = *reinterpret_cast<const uint4 *>(row + r * row_stride + 16 * c);
                const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int wi = 0; wi < 4; ++wi) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&u[wi]));
                    dot[r] = fmaf(f.x, mv[2 * wi], dot[r]);
                    dot[r] = fmaf(f.y, mv[2 * wi + 1], dot[r]);
                    nn[r] = fmaf(f.x, f.x, nn[r]);
                    nn[r] = fmaf(f.y, f.y, nn[r]);
                }
            }
        }
    }
}

// Pass 2: persistent CTA, blocks blockIdx.x + i * gridDim.x through a ring
// of KD_STAGES stages.  A producer warp (one lane) copies a block's
// descriptor and stretches into a stage once every consumer warp has
// released it (empty barrier, one arrival per warp); consumers wait on the
// stage's full barrier.  Consumer warp w takes slabs of 2 * RG rows (RG =
// max(1, 32 / Hk)): lane t of a pass scores rows t / Hk and t / Hk + RG of
// head t % Hk, reading the head's mean once for both.  The f16 means sit in
// shared memory with rows padded by one float4 (D / 4 + 1 chunks, odd),
// which spreads the lanes' reads over the banks; the q8_0 digit planes of a
// head are 3 * D bytes apart.
template <bool Q8, int D>
__global__ void __launch_bounds__((KD_SCORE_WARPS + 1) * 32, 1)
    keydiff_score_kernel(const __grid_constant__ KeyDiffArgs a) {
    constexpr int MS = D + 4;
    extern __shared__ __align__(128) uint8_t smem[];
    const int Hk = a.Hk;
    const Geom G = geom(Q8, D, a.block_rows);
    const int stage_bytes = Hk * (G.hsb + G.srs);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + KD_STAGES;
    KeyDiffBlock *sdesc = reinterpret_cast<KeyDiffBlock *>(smem + 64);
    uint8_t *stages = smem + 128;
    uint8_t *smeanb = stages + (size_t)KD_STAGES * stage_bytes;
    float *smean = reinterpret_cast<float *>(smeanb);            // f16: [Hk][MS]
    int8_t *sdig = reinterpret_cast<int8_t *>(smeanb);           // q8_0: [Hk][3][D]
    float *snorm = reinterpret_cast<float *>(smeanb + score_mean_bytes(Q8, Hk, D));
    float *sstep = snorm + Hk;                                   // q8_0: ms per head
    const int rg = Hk >= 32 ? 1 : 32 / Hk, items = rg * Hk, passes = (items + 31) / 32;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const bool producer = w == KD_SCORE_WARPS;
    auto issue = [&](int s, int b) {
        const KeyDiffBlock bk = a.blocks[b];
        sdesc[s] = bk;
        uint8_t *st = stages + (size_t)s * stage_bytes;
        uint32_t bytes = 0;
        for (int g = 0; g < Hk; ++g)
            bytes += issue_head(a, G, bk, g, st + g * G.hsb, st + Hk * G.hsb + g * G.srs, &full[s], false);
        mbar_expect_tx(&full[s], bytes);
        for (int g = 0; g < Hk; ++g)
            issue_head(a, G, bk, g, st + g * G.hsb, st + Hk * G.hsb + g * G.srs, &full[s], true);
    };
    if (producer && lane == 0) {
        for (int s = 0; s < KD_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], KD_SCORE_WARPS);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int s = 0; s < KD_STAGES; ++s)
            if (blockIdx.x + s * gridDim.x < a.n_blocks) issue(s, blockIdx.x + s * gridDim.x);
    }
    for (int i = threadIdx.x; i < Hk; i += blockDim.x) snorm[i] = a.mean_norm[i];
    if constexpr (Q8) {
        // per head: ms = max |mu| / QMAX (warp w takes heads w, w + warps, ...)
        for (int g = w; g < Hk; g += KD_SCORE_WARPS + 1) {
            float mx = 0.f;
            for (int d = lane; d < D; d += 32) mx = fmaxf(mx, fabsf(a.mean[g * D + d]));
            for (int m = 16; m > 0; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
            if (lane == 0) sstep[g] = mx / (float)QMAX;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < Hk * D; i += blockDim.x) {
            const int g = i / D, d = i % D;
            const float ms = sstep[g];
            int q = ms > 0.f ? __float2int_rn(a.mean[i] / ms) : 0;
            q = max(-QMAX, min(QMAX, q));
            const int lo = ((q + 128) & 255) - 128;
            const int q1 = (q - lo) >> 8;
            const int mid = ((q1 + 128) & 255) - 128;
            const int hi = (q1 - mid) >> 8;
            sdig[(g * 3 + 0) * D + d] = (int8_t)hi;
            sdig[(g * 3 + 1) * D + d] = (int8_t)mid;
            sdig[(g * 3 + 2) * D + d] = (int8_t)lo;
        }
    } else {
        for (int i = threadIdx.x; i < Hk * D; i += blockDim.x) smean[(i / D) * MS + i % D] = a.mean[i];
    }
    __syncthreads();
    if (producer) {
        if (lane != 0) return;
        int it = KD_STAGES;
        for (int64_t b = blockIdx.x + (int64_t)KD_STAGES * gridDim.x; b < a.n_blocks; b += gridDim.x, ++it) {
            const int s = it % KD_STAGES;
            if (!mbar_wait_bounded(&empty[s], (unsigned)(it / KD_STAGES - 1) & 1u)) {
                atomicOr(a.err, ERR_WAIT_TIMEOUT);
                for (int k = 1; k <= KD_STAGES; ++k) { // the copies still in flight
                    const int it2 = it - k;
                    if (blockIdx.x + (int64_t)it2 * gridDim.x < a.n_blocks)
                        mbar_wait_bounded(&full[it2 % KD_STAGES], (unsigned)(it2 / KD_STAGES) & 1u);
                }
                return;
            }
            issue(s, (int)b);
        }
        return;
    }
    const int CHR = (Q8 ? D : 2 * D) / 16;
    const int rot = CHR == 4 ? ((lane >> 1) & 3) : (lane & 7);
    float *sterm = sstep + Hk + w * 2 * items;
    int it = 0;
    for (int b = blockIdx.x; b < a.n_blocks; b += gridDim.x, ++it) {
        const int s = it % KD_STAGES;
        if (!mbar_wait_bounded(&full[s], (unsigned)(it / KD_STAGES) & 1u)) {
            if (lane == 0) atomicOr(a.err, ERR_WAIT_TIMEOUT);
            return;
        }
        const KeyDiffBlock bk = sdesc[s];
        const uint8_t *st = stages + (size_t)s * stage_bytes;
        for (int r0 = w * 2 * rg; r0 < bk.n; r0 += KD_SCORE_WARPS * 2 * rg) {
            for (int p = 0; p < passes; ++p) {
                const int t = p * 32 + lane, rr = t / Hk, g = t % Hk;
                if (t >= items || r0 + rr >= bk.n) continue;
                // rows r0 + rr and r0 + rr + rg; past the block's end the second is the first again (its
                // terms land in a slot nobody reads)
                const bool two = r0 + rr + rg < bk.n;
                const int64_t row = bk.row0 + a.layer_off + (int64_t)g * a.P;
                const uint8_t *sc =
                    Q8 ? st + Hk * G.hsb + g * G.srs + scale_skew(a, row, G.sb) + (r0 + rr) * G.sb : nullptr;
                float dot[2], nn[2];
                row_terms<Q8, D, 2>(st + g * G.hsb + (r0 + rr) * G.rb, two ? rg * G.rb : 0, sc, two ? rg * G.sb : 0,
                                    smean + g * MS, sdig + g * 3 * D, rot, dot, nn);
                const float mn = snorm[g];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float dr = Q8 ? dot[r] * sstep[g] : dot[r];
                    const float cs = (nn[r] > 0.f && mn > 0.f) ? dr / (sqrtf(nn[r]) * mn) : 0.f; // degenerate: 0
                    sterm[(r * rg + rr) * Hk + g] = 1.f - cs;
                }
            }
            __syncwarp();
            if (lane < 2 * rg && r0 + lane < bk.n) {
                float score = 0.f;
                for (int g = 0; g < Hk; ++g) score += sterm[lane * Hk + g];
                a.score[bk.i0 + r0 + lane] = score / (float)Hk;
            }
            __syncwarp();
        }
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&empty[s])) : "memory");
    }
}

template <bool Q8, int D>
cudaError_t launch_typed(const KeyDiffArgs &a, int sms, cudaStream_t st) {
    const Geom G = geom(Q8, D, a.block_rows);
    const size_t sum_smem = std::max<size_t>((size_t)KD_WARPS * (G.hsb + G.srs), (size_t)KD_WARPS * 32 * 16 * 4);
    const size_t score_sm = score_smem(Q8, a.Hk, D, a.block_rows);
    if (sum_smem > KD_SMEM_MAX || score_sm > KD_SMEM_MAX) return cudaErrorInvalidValue;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(keydiff_sum_kernel<Q8, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)sum_smem)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(keydiff_score_kernel<Q8, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)score_sm)) != cudaSuccess)
        return e;
    keydiff_sum_kernel<Q8, D><<<(unsigned)(a.Hk * a.n_slices), KD_WARPS * 32, sum_smem, st>>>(a);
    keydiff_mean_kernel<<<(unsigned)a.Hk, 1024u, 0, st>>>(a);
    const unsigned grid = (unsigned)std::min<int64_t>(a.n_blocks, (int64_t)sms);
    keydiff_score_kernel<Q8, D><<<grid, (KD_SCORE_WARPS + 1) * 32, score_sm, st>>>(a);
    return cudaGetLastError();
}

} // namespace

int keydiff_block_rows(bool q8, int Hk, int D) {
    for (int br = 64; br > 1; --br)
        if (score_smem(q8, Hk, D, br) <= (size_t)KD_SMEM_MAX - 1024) return br;
    return 1;
}

int keydiff_slice_blocks() {
    return KD_WARPS;
}

cudaError_t launch_keydiff(const KeyDiffArgs &a, int sms, cudaStream_t st) {
    if (a.n_rows <= 0 || a.n_blocks <= 0) return cudaSuccess;
    if (a.D != 64 && a.D != 128) return cudaErrorInvalidValue;
    if (a.q8) return a.D == 128 ? launch_typed<true, 128>(a, sms, st) : launch_typed<true, 64>(a, sms, st);
    return a.D == 128 ? launch_typed<false, 128>(a, sms, st) : launch_typed<false, 64>(a, sms, st);
}

} // namespace kvc
