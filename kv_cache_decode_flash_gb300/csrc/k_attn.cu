// k_attn.cu - single-token decode attention over a q8_0 or f16 grouped-query
// KV cache, split-K over KV chunks with an online-softmax merge.
//
// What is computed: out[h] = softmax_j(kq_scale * q[h] . K_j) V_j for every
// row j of the sequence, query head h reading KV head h / r (grouped-query
// heads stay in whole KV-head groups: "F5 - Advanced KV Cache Techniques",
// sections M2 - HeadInfer and M3 - NEO, the gpu_heads * gqa_ratio split).
// Partial results of KV chunks are combined with the online-softmax rule
// (same page, section M4 - ScoutAttention: merge via FlashAttention's
// online-softmax merge; section F5-opt W4: inter-tile online softmax).
//
// Layout of the work: grid (chunk, kv head).  A CTA streams its chunk in
// tiles of 128 rows through a multi-stage shared-memory ring filled by TMA
// (K and V rows as 2-D boxes of 16 rows, K with the 128-/64-byte swizzle so
// the tensor-core fragment loads are bank-conflict free; q8_0 scales by
// 1-D bulk copies).  Each of the 8 warps owns 16 rows of every tile and runs
// its own online softmax:
//   QK  on the tensor cores (mma.sync m16n8k16, fp32 accumulate): int8 codes
//       become exact fp16 values in registers, q is split into fp16 hi + lo
//       parts (about 22 significant bits), and each 32-element block gets its
//       own accumulator so the block scale is applied in fp32 afterwards;
//   PV  on the CUDA cores with packed fp32x2 FMAs (fp32 accumulate); the
//       q8_0 V scale is folded into the probability (p * d_v per block).
// Warps merge inside the CTA; CTAs of one (sequence, kv head) merge through
// global partials, the last CTA to arrive (an atomic ticket, no waiting)
// combining them in fixed chunk order, so results are bitwise repeatable.
#include "kvc_internal.h"

#include <cuda_fp16.h>

namespace kvc {
namespace {

constexpr uint32_t WAIT_LIMIT = 1u << 24;

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
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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
// Bounded wait: gives up after WAIT_LIMIT polls and reports it in *err.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity, uint32_t *err) {
    for (uint32_t i = 0; i < WAIT_LIMIT; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    atomicOr(err, ERR_WAIT_TIMEOUT);
    return false;
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void bulk_load(void *dst, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four int8 codes -> two half2 of their exact values: (c0,c1) and (c2,c3).
// Bytes are flipped to offset binary u = c + 128 and placed in the low
// mantissa byte of 0x64xx (= 1024 + u); subtracting 1152 gives c exactly.
__device__ __forceinline__ void codes_to_half2(uint32_t w, uint32_t &h01, uint32_t &h23) {
    const uint32_t u = w ^ 0x80808080u;
    asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(h01) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(h23) : "r"(u), "r"(0x64646464u));
    const uint32_t bias = 0x64806480u; // half2(1152, 1152)
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(h01) : "r"(bias));
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(h23) : "r"(bias));
}

// Eight int8 codes (two words) -> eight fp32 values, as four float2.
// Each byte goes into the low mantissa byte of 2^23 (0x4B0000xx = 2^23 + u);
// subtracting 2^23 + 128 gives the signed code exactly.
__device__ __forceinline__ void codes_to_f32x8(uint32_t w0, uint32_t w1, float2 (&v)[4]) {
    const uint32_t u0 = w0 ^ 0x80808080u, u1 = w1 ^ 0x80808080u;
    const uint32_t mag = 0x4B000000u;
    uint32_t f[8];
    asm("prmt.b32 %0, %1, %2, 0x7650;" : "=r"(f[0]) : "r"(u0), "r"(mag));
    asm("prmt.b32 %0, %1, %2, 0x7651;" : "=r"(f[1]) : "r"(u0), "r"(mag));
    asm("prmt.b32 %0, %1, %2, 0x7652;" : "=r"(f[2]) : "r"(u0), "r"(mag));
    asm("prmt.b32 %0, %1, %2, 0x7653;" : "=r"(f[3]) : "r"(u0), "r"(mag));
    asm("prmt.b32 %0, %1, %2, 0x7650;" : "=r"(f[4]) : "r"(u1), "r"(mag));
    asm("prmt.b32 %0, %1, %2, 0x7651;" : "=r"(f[5]) : "r"(u1), "r"(mag));
    asm("prmt.b32 %0, %1, %2, 0x7652;" : "=r"(f[6]) : "r"(u1), "r"(mag));
    asm("prmt.b32 %0, %1, %2, 0x7653;" : "=r"(f[7]) : "r"(u1), "r"(mag));
    const float b = 8388736.0f; // 2^23 + 128
    const float2 bb = make_float2(b, b);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 x = make_float2(__uint_as_float(f[2 * i]), __uint_as_float(f[2 * i + 1]));
        unsigned long long xr = *reinterpret_cast<unsigned long long *>(&x);
        unsigned long long br = *reinterpret_cast<const unsigned long long *>(&bb);
        asm("sub.rn.f32x2 %0, %0, %1;" : "+l"(xr) : "l"(br));
        v[i] = *reinterpret_cast<float2 *>(&xr);
    }
}

__device__ __forceinline__ void fma2(float2 &acc, const float2 a, const float2 b) {
    unsigned long long ar = *reinterpret_cast<const unsigned long long *>(&a);
    unsigned long long br = *reinterpret_cast<const unsigned long long *>(&b);
    unsigned long long cr = *reinterpret_cast<unsigned long long *>(&acc);
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(cr) : "l"(ar), "l"(br));
    acc = *reinterpret_cast<float2 *>(&cr);
}

__device__ __forceinline__ void mul2(float2 &acc, const float2 a) {
    unsigned long long ar = *reinterpret_cast<const unsigned long long *>(&a);
    unsigned long long cr = *reinterpret_cast<unsigned long long *>(&acc);
    asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(cr) : "l"(ar));
    acc = *reinterpret_cast<float2 *>(&cr);
}


// Four int8 codes -> four fp32 values (two float2), exact (see codes_to_f32x8).
__device__ __forceinline__ void codes_to_f32x4(uint32_t w, float2 (&v)[2]) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t mag = 0x4B000000u;
    uint32_t f[4];
    asm("prmt.b32 %0, %1, %2, 0x7650;" : "=r"(f[0]) : "r"(u), "r"(mag));
    asm("prmt.b32 %0, %1, %2, 0x7651;" : "=r"(f[1]) : "r"(u), "r"(mag));
    asm("prmt.b32 %0, %1, %2, 0x7652;" : "=r"(f[2]) : "r"(u), "r"(mag));
    asm("prmt.b32 %0, %1, %2, 0x7653;" : "=r"(f[3]) : "r"(u), "r"(mag));
    const float b = 8388736.0f; // 2^23 + 128
    const float2 bb = make_float2(b, b);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        float2 x = make_float2(__uint_as_float(f[2 * i]), __uint_as_float(f[2 * i + 1]));
        unsigned long long xr = *reinterpret_cast<unsigned long long *>(&x);
        unsigned long long br = *reinterpret_cast<const unsigned long long *>(&bb);
        asm("sub.rn.f32x2 %0, %0, %1;" : "+l"(xr) : "l"(br));
        v[i] = *reinterpret_cast<float2 *>(&xr);
    }
}

// Programmatic dependent launch: wait for the preceding kernel's results /
// let the next kernel be scheduled.  No-ops without a programmatic edge.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Static shape of one kernel instance.  W warps per CTA, each owning 16 rows
// of every tile; stages sized so two CTAs fit on an SM.
template <int TYPE, int D, int R>
struct Shape {
    static constexpr bool Q8 = TYPE == KVC_Q8_0;
    static constexpr int W = Q8 ? 8 : 4;              // warps per CTA
    static constexpr int T = 16 * W;                  // rows per tile
    static constexpr int NB = D / 32;                 // q8_0 blocks per row
    static constexpr int KROW = Q8 ? D : 2 * D;       // bytes per K row
    static constexpr int VROW = KROW;                 // bytes per V row
    static constexpr int SB = Q8 ? NB * 2 : 0;        // scale bytes per row
    static constexpr int KSUB = Q8 ? 1 : (D == 128 ? 2 : 1); // f16 K sub-tiles of 64 halves
    static constexpr int SCALE_BUF = Q8 ? ((T * SB + 32 + 127) / 128) * 128 : 0;
    static constexpr int KBYTES = T * KROW, VBYTES = T * VROW;
    static constexpr int STAGE = ((KBYTES + VBYTES + 2 * SCALE_BUF + 1023) / 1024) * 1024; // 1024-aligned stages
    static constexpr int KSTEPS = D / 16;
    static constexpr int NBX = Q8 ? NB : 1;           // probability blocks per row
    static constexpr int RP = 4 * ((R + 1) / 2);      // floats per (row, block) in the exchange
    static constexpr int PROW = NBX * RP + 4;         // floats per row in the exchange
    static constexpr int PBUF = 16 * PROW;            // floats per warp
    // as many stages (2..4) as fit in 110 KiB with the exchange buffers: two CTAs per SM
    static constexpr int FIT = (110 * 1024 - W * PBUF * 4 - 2048) / STAGE;
    static constexpr int STAGES = FIT < 2 ? 2 : (FIT > 4 ? 4 : FIT);
    static constexpr int LPR = D / 4;                 // PV lanes per row (4 dims per lane)
    static constexpr int RPS = 32 / LPR;              // PV rows per step
    static constexpr int OOFF = ((2 * R + 3) / 4) * 4;  // partial: m[R], l[R], pad, then o[R][D] 16-byte aligned
    static constexpr int PF = OOFF + R * D;            // floats of one partial
    static constexpr int SMEM = STAGES * STAGE + W * PBUF * 4 + W * 16 * 4 + 2 * STAGES * 8 + 64 + 1024;
    static constexpr int MINB = Q8 ? 2 : 4;           // CTAs per SM the register budget targets
    static constexpr int MERGE_CAP = (STAGES * STAGE) / (8 * R); // chunks the grid merge can stage
};

// Byte offset of 16-byte chunk `c` of row `row` in a TMA-swizzled K tile.
template <int ROWB>
__device__ __forceinline__ int swz(int row, int c) {
    if constexpr (ROWB == 128)
        return row * 128 + ((c ^ (row & 7)) << 4);
    else
        return row * 64 + ((c ^ ((row >> 1) & 3)) << 4);
}

struct TileInfo {
    int n;     // rows in the tile
    int delta; // scale rows skipped by the 16-byte alignment of the scale copy
};

template <int TYPE, int D, int R>
__global__ void __launch_bounds__(Shape<TYPE, D, R>::W * 32, Shape<TYPE, D, R>::MINB)
    attn_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmk,
                const __grid_constant__ CUtensorMap tmv) {
    using S = Shape<TYPE, D, R>;
    constexpr int W = S::W, T = S::T, NT = W * 32;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *stages = smem;
    float *pbuf_all = reinterpret_cast<float *>(smem + S::STAGES * S::STAGE);
    float *abuf_all = pbuf_all + W * S::PBUF;
    uint64_t *full = reinterpret_cast<uint64_t *>(abuf_all + W * 16);
    uint64_t *empty = full + S::STAGES;
    TileInfo *tinfo = reinterpret_cast<TileInfo *>(empty + S::STAGES);
    __shared__ int s_flag;
    __shared__ float s_M[R], s_L[R];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = blockIdx.y;
    const int chunk = blockIdx.x;

    // ---- which sequence / chunk (parameters only: safe before the wait) ----
    int si = 0;
    for (int i = 1; i < p.n_seq; ++i)
        if (chunk >= p.seq[i].chunk0) si = i;
    const AttnSeq sq = p.seq[si];
    const int lc = chunk - sq.chunk0;
    const int r_act = p.r;
    const int row_begin = lc * p.chunk_rows;
    const int row_end = min(sq.n_rows, row_begin + p.chunk_rows);

    // tiles never cross a page: their sizes follow from (off, rows, P) alone
    auto tile_rows = [&](int r0) { return min(min(T, row_end - r0), p.P - (sq.off + r0) % p.P); };
    int n_tiles = 0;
    for (int r0 = row_begin; r0 < row_end; r0 += tile_rows(r0)) ++n_tiles;

    if (tid == 0) {
        for (int s = 0; s < S::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], W);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // ---- producer (thread 0) -----------------------------------------------
    int prod_r0 = row_begin, prod_k = 0;
    auto issue = [&](int k) {
        const int s = k % S::STAGES;
        const int n = tile_rows(prod_r0);
        const int lr = sq.off + prod_r0;
        const int page = sq.page_table[lr / p.P];
        const int cell = lr % p.P;
        prod_r0 += n;
        const int64_t R0 = ((int64_t)page * p.Hk + g) * p.P + cell;
        uint8_t *st = stages + s * S::STAGE;
        const int nb = (n + TMA_BOX_ROWS - 1) / TMA_BOX_ROWS;
        unsigned bytes = (unsigned)(nb * TMA_BOX_ROWS * (S::KROW + S::VROW));
        int delta = 0;
        unsigned sbytes = 0;
        int64_t saligned = 0;
        if constexpr (S::Q8) {
            const int64_t start = R0 * S::SB;
            saligned = start & ~(int64_t)15;
            delta = (int)((start - saligned) / S::SB);
            const int64_t end = (start + (int64_t)n * S::SB + 15) & ~(int64_t)15;
            sbytes = (unsigned)(end - saligned);
            if (saligned + (int64_t)sbytes > p.scale_limit_bytes) {
                atomicOr(p.err, ERR_BAD_INDEX);
                sbytes = 0;
            }
            bytes += 2 * sbytes;
        }
        tinfo[s].n = n;
        tinfo[s].delta = delta;
        mbar_expect_tx(&full[s], bytes);
        for (int b = 0; b < nb; ++b) {
            const int y = (int)(R0 + b * TMA_BOX_ROWS);
            if constexpr (S::Q8 || S::KSUB == 1) {
                tma_load_2d(st + b * TMA_BOX_ROWS * (S::Q8 ? S::KROW : 128), &tmk, 0, y, &full[s]);
            } else {
                tma_load_2d(st + b * TMA_BOX_ROWS * 128, &tmk, 0, y, &full[s]);
                tma_load_2d(st + T * 128 + b * TMA_BOX_ROWS * 128, &tmk, 64, y, &full[s]);
            }
            tma_load_2d(st + S::KBYTES + b * TMA_BOX_ROWS * S::VROW, &tmv, 0, y, &full[s]);
        }
        if constexpr (S::Q8) {
            if (sbytes) {
                bulk_load(st + S::KBYTES + S::VBYTES, reinterpret_cast<const uint8_t *>(p.ks) + saligned, sbytes,
                          &full[s]);
                bulk_load(st + S::KBYTES + S::VBYTES + S::SCALE_BUF,
                          reinterpret_cast<const uint8_t *>(p.vs) + saligned, sbytes, &full[s]);
            }
        }
    };
    // Tiles made only of rows no in-flight kernel writes (the stable prefix)
    // are requested before waiting for the preceding kernel.
    if (tid == 0) {
        while (prod_k < n_tiles && prod_k < S::STAGES && prod_r0 + tile_rows(prod_r0) <= sq.stable_rows)
            issue(prod_k++);
    }
    pdl_wait();
    pdl_trigger();
    if (tid == 0) {
        for (; prod_k < n_tiles && prod_k < S::STAGES; ++prod_k) issue(prod_k);
    }

    // ---- query fragments (B operand of QK), hi + lo fp16 -------------------
    const int gq = lane >> 2, tq = lane & 3;
    const int hslot = gq; // head slot this lane feeds into the MMA B operand
    const bool hvalid = hslot < r_act;
    const float *qrow = p.q + ((int64_t)sq.out_row * p.H + (int64_t)g * r_act + (hvalid ? hslot : 0)) * D;
    float qv[S::KSTEPS][4];
    float amax = 0.0f;
#pragma unroll
    for (int ks = 0; ks < S::KSTEPS; ++ks) {
        int d0, d1;
        if constexpr (S::Q8) {
            d0 = 16 * ks + 4 * tq;
            d1 = d0 + 2;
        } else {
            d0 = 16 * ks + 2 * tq;
            d1 = d0 + 8;
        }
        float2 x0 = hvalid ? *reinterpret_cast<const float2 *>(qrow + d0) : make_float2(0.f, 0.f);
        float2 x1 = hvalid ? *reinterpret_cast<const float2 *>(qrow + d1) : make_float2(0.f, 0.f);
        qv[ks][0] = x0.x * p.kq_scale_log2;
        qv[ks][1] = x0.y * p.kq_scale_log2;
        qv[ks][2] = x1.x * p.kq_scale_log2;
        qv[ks][3] = x1.y * p.kq_scale_log2;
#pragma unroll
        for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fabsf(qv[ks][j]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    // power-of-two scaling that puts max|q| in [2^13, 2^14): hi and lo stay normal fp16
    const int e_q = (amax > 0.0f) ? 13 - ilogbf(amax) : 0;
    uint32_t bh[S::KSTEPS][2], bl[S::KSTEPS][2];
#pragma unroll
    for (int ks = 0; ks < S::KSTEPS; ++ks) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float x0 = ldexpf(qv[ks][2 * j], e_q), x1 = ldexpf(qv[ks][2 * j + 1], e_q);
            const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
            const __half l0 = __float2half_rn(x0 - __half2float(h0)), l1 = __float2half_rn(x1 - __half2float(h1));
            bh[ks][j] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
            bl[ks][j] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
        }
    }
    // 2^-e for the two heads (2t, 2t+1) whose scores this lane accumulates
    const int e0 = __shfl_sync(0xffffffffu, e_q, (2 * tq) * 4);
    const int e1 = __shfl_sync(0xffffffffu, e_q, (2 * tq + 1) * 4);
    const float hs0 = ldexpf(1.0f, -e0), hs1 = ldexpf(1.0f, -e1);
    const bool hv0 = 2 * tq < r_act, hv1 = 2 * tq + 1 < r_act;

    // ---- per-warp online-softmax state -------------------------------------
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f; // heads 2t, 2t+1
    float2 o[R][2];
#pragma unroll
    for (int h = 0; h < R; ++h)
#pragma unroll
        for (int j = 0; j < 2; ++j) o[h][j] = make_float2(0.f, 0.f);
    float *pbuf = pbuf_all + warp * S::PBUF;
    float *abuf = abuf_all + warp * 16;
    const int rbase = warp * 16;
    const int pv_ro = lane / S::LPR, pv_d0 = 4 * (lane % S::LPR);
    const int pv_b = S::Q8 ? pv_d0 / 32 : 0;

    for (int k = 0; k < n_tiles; ++k) {
        const int s = k % S::STAGES;
        if (!mbar_wait(&full[s], (k / S::STAGES) & 1, p.err)) break;
        const uint8_t *st = stages + s * S::STAGE;
        const int n = tinfo[s].n;
        const int rows_w = min(max(n - rbase, 0), 16);
        if (rows_w > 0) {
            // ---------------- QK on the tensor cores ----------------
            float sc[4] = {0.f, 0.f, 0.f, 0.f}; // (row g, 2t) (row g, 2t+1) (row g+8, 2t) (row g+8, 2t+1)
            const int ra = rbase + gq, rb = ra + 8;
            if constexpr (S::Q8) {
                const uint16_t *ksc = reinterpret_cast<const uint16_t *>(st + S::KBYTES + S::VBYTES) +
                                      tinfo[s].delta * S::NB;
#pragma unroll
                for (int b = 0; b < S::NB; ++b) {
                    float ch[4] = {0.f, 0.f, 0.f, 0.f}, cl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int s2 = 0; s2 < 2; ++s2) {
                        const int ks = 2 * b + s2;
                        const uint32_t wa = *reinterpret_cast<const uint32_t *>(st + swz<S::KROW>(ra, ks) + 4 * tq);
                        const uint32_t wb = *reinterpret_cast<const uint32_t *>(st + swz<S::KROW>(rb, ks) + 4 * tq);
                        uint32_t a0, a1, a2, a3;
                        codes_to_half2(wa, a0, a2);
                        codes_to_half2(wb, a1, a3);
                        mma16816(ch, a0, a1, a2, a3, bh[ks][0], bh[ks][1]);
                        mma16816(cl, a0, a1, a2, a3, bl[ks][0], bl[ks][1]);
                    }
                    const float da = __half2float(__ushort_as_half(ksc[ra * S::NB + b]));
                    const float db = __half2float(__ushort_as_half(ksc[rb * S::NB + b]));
                    sc[0] = fmaf(da, ch[0] + cl[0], sc[0]);
                    sc[1] = fmaf(da, ch[1] + cl[1], sc[1]);
                    sc[2] = fmaf(db, ch[2] + cl[2], sc[2]);
                    sc[3] = fmaf(db, ch[3] + cl[3], sc[3]);
                }
            } else {
                float ch[4] = {0.f, 0.f, 0.f, 0.f}, cl[4] = {0.f, 0.f, 0.f, 0.f};
                const int lrow = rbase + (lane & 15);
#pragma unroll
                for (int ks = 0; ks < S::KSTEPS; ++ks) {
                    const int sub = ks / 4;
                    const int c = 2 * (ks % 4) + (lane >> 4);
                    const uint32_t addr = smem_u32(st + sub * T * 128 + swz<128>(lrow, c));
                    uint32_t a0, a1, a2, a3;
                    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                                 : "r"(addr));
                    mma16816(ch, a0, a1, a2, a3, bh[ks][0], bh[ks][1]);
                    mma16816(cl, a0, a1, a2, a3, bl[ks][0], bl[ks][1]);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) sc[j] = ch[j] + cl[j];
            }
            // log2-domain scores; rows beyond the tile are -inf
            float s2v[4];
            s2v[0] = (gq < rows_w) ? sc[0] * hs0 : -INFINITY;
            s2v[1] = (gq < rows_w) ? sc[1] * hs1 : -INFINITY;
            s2v[2] = (gq + 8 < rows_w) ? sc[2] * hs0 : -INFINITY;
            s2v[3] = (gq + 8 < rows_w) ? sc[3] * hs1 : -INFINITY;
            // ---------------- online softmax (per warp) ----------------
            float t0 = fmaxf(s2v[0], s2v[2]), t1 = fmaxf(s2v[1], s2v[3]);
#pragma unroll
            for (int m = 4; m < 32; m <<= 1) {
                t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, m));
                t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, m));
            }
            const float mn0 = fmaxf(m0, t0), mn1 = fmaxf(m1, t1);
            const float al0 = (mn0 == -INFINITY) ? 1.f : exp2f(m0 - mn0);
            const float al1 = (mn1 == -INFINITY) ? 1.f : exp2f(m1 - mn1);
            float pr[4];
            pr[0] = (hv0 && s2v[0] != -INFINITY) ? exp2f(s2v[0] - mn0) : 0.f;
            pr[1] = (hv1 && s2v[1] != -INFINITY) ? exp2f(s2v[1] - mn1) : 0.f;
            pr[2] = (hv0 && s2v[2] != -INFINITY) ? exp2f(s2v[2] - mn0) : 0.f;
            pr[3] = (hv1 && s2v[3] != -INFINITY) ? exp2f(s2v[3] - mn1) : 0.f;
            float rs0 = pr[0] + pr[2], rs1 = pr[1] + pr[3];
#pragma unroll
            for (int m = 4; m < 32; m <<= 1) {
                rs0 += __shfl_xor_sync(0xffffffffu, rs0, m);
                rs1 += __shfl_xor_sync(0xffffffffu, rs1, m);
            }
            l0 = l0 * al0 + rs0;
            l1 = l1 * al1 + rs1;
            m0 = mn0;
            m1 = mn1;
            // ---------------- exchange: p * d_v per block, duplicated in pairs ----
            if (4 * tq < S::RP) {
                const uint16_t *vsc =
                    S::Q8 ? reinterpret_cast<const uint16_t *>(st + S::KBYTES + S::VBYTES + S::SCALE_BUF) +
                                tinfo[s].delta * S::NB
                          : nullptr;
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int row = gq + 8 * hr; // row within the warp's 16
                    const float pa = pr[2 * hr], pb = pr[2 * hr + 1];
                    const bool live = row < rows_w;
#pragma unroll
                    for (int b = 0; b < S::NBX; ++b) {
                        float dv = 1.f;
                        if constexpr (S::Q8) dv = live ? __half2float(__ushort_as_half(vsc[(rbase + row) * S::NB + b])) : 0.f;
                        const float xa = live ? pa * dv : 0.f, xb = live ? pb * dv : 0.f;
                        *reinterpret_cast<float4 *>(pbuf + row * S::PROW + b * S::RP + 4 * tq) =
                            make_float4(xa, xa, xb, xb);
                    }
                }
            }
            if (gq == 0) {
                abuf[2 * tq] = al0;
                abuf[2 * tq + 1] = al1;
            }
            __syncwarp();
            // ---------------- rescale and PV on the CUDA cores ----------------
            float2 al[R];
            bool any = false;
#pragma unroll
            for (int h = 0; h < R; ++h) {
                const float a = abuf[h];
                al[h] = make_float2(a, a);
                any |= (a != 1.f);
            }
            if (any) {
#pragma unroll
                for (int h = 0; h < R; ++h)
#pragma unroll
                    for (int j = 0; j < 2; ++j) mul2(o[h][j], al[h]);
            }
            const uint8_t *vt = st + S::KBYTES;
#pragma unroll 4
            for (int r0 = 0; r0 < rows_w; r0 += S::RPS) {
                const int row = r0 + pv_ro;
                float2 vv[2];
                if constexpr (S::Q8) {
                    const uint32_t w = *reinterpret_cast<const uint32_t *>(vt + (rbase + row) * S::VROW + pv_d0);
                    codes_to_f32x4(w, vv);
                } else {
                    const uint2 w2 = *reinterpret_cast<const uint2 *>(vt + (rbase + row) * S::VROW + 2 * pv_d0);
                    vv[0] = __half22float2(*reinterpret_cast<const __half2 *>(&w2.x));
                    vv[1] = __half22float2(*reinterpret_cast<const __half2 *>(&w2.y));
                }
                const float *pp = pbuf + row * S::PROW + pv_b * S::RP;
#pragma unroll
                for (int hp = 0; hp < (R + 1) / 2; ++hp) {
                    const float4 q4 = *reinterpret_cast<const float4 *>(pp + 4 * hp);
                    const float2 pa = make_float2(q4.x, q4.y), pb = make_float2(q4.z, q4.w);
                    fma2(o[2 * hp][0], pa, vv[0]);
                    fma2(o[2 * hp][1], pa, vv[1]);
                    if (2 * hp + 1 < R) {
                        fma2(o[2 * hp + 1][0], pb, vv[0]);
                        fma2(o[2 * hp + 1][1], pb, vv[1]);
                    }
                }
            }
        }
        // release the stage; thread 0 refills it once every warp is done
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (tid == 0 && prod_k < n_tiles) {
            const int ps = prod_k % S::STAGES;
            if (mbar_wait(&empty[ps], ((prod_k / S::STAGES) - 1) & 1, p.err)) issue(prod_k);
            ++prod_k;
        }
    }
    // drain: make sure no copy is still landing in shared memory before reuse
    if (tid == 0) {
        for (int k = max(0, prod_k - S::STAGES); k < prod_k; ++k) {
            const int s = k % S::STAGES;
            mbar_wait(&full[s], (k / S::STAGES) & 1, p.err);
        }
    }
    __syncthreads();

    // ---- reduce the row-parallel lanes of each warp ----------------------------
#pragma unroll
    for (int m = S::LPR; m < 32; m <<= 1)
#pragma unroll
        for (int h = 0; h < R; ++h)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                o[h][j].x += __shfl_xor_sync(0xffffffffu, o[h][j].x, m);
                o[h][j].y += __shfl_xor_sync(0xffffffffu, o[h][j].y, m);
            }
    // ---- CTA merge of the warps (stages are free now) -------------------------
    float *wm = reinterpret_cast<float *>(stages); // [W][R]
    float *wl = wm + W * R;                         // [W][R]
    float *wo = wl + W * R;                         // [W][R][D]
    if (gq == 0) {
        if (2 * tq < R) {
            wm[warp * R + 2 * tq] = m0;
            wl[warp * R + 2 * tq] = l0;
        }
        if (2 * tq + 1 < R) {
            wm[warp * R + 2 * tq + 1] = m1;
            wl[warp * R + 2 * tq + 1] = l1;
        }
    }
    if (lane < S::LPR) {
#pragma unroll
        for (int h = 0; h < R; ++h) {
            float4 v4 = make_float4(o[h][0].x, o[h][0].y, o[h][1].x, o[h][1].y);
            *reinterpret_cast<float4 *>(wo + (warp * R + h) * D + pv_d0) = v4;
        }
    }
    __syncthreads();

    const int n_chunks = sq.n_chunks;
    float *part = p.part + ((int64_t)chunk * p.Hk + g) * S::PF;
    float *outp = p.out + ((int64_t)sq.out_row * p.H + (int64_t)g * r_act) * D;
    for (int idx = tid; idx < r_act * D; idx += NT) {
        const int h = idx / D, i = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < W; ++w) M = fmaxf(M, wm[w * R + h]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            const float f = (M == -INFINITY) ? 0.f : exp2f(wm[w * R + h] - M);
            L += wl[w * R + h] * f;
            O += wo[(w * R + h) * D + i] * f;
        }
        if (n_chunks == 1) {
            outp[h * D + i] = (L > 0.f) ? O / L : 0.f;
        } else {
            if (i == 0) {
                part[h] = M;
                part[R + h] = L;
            }
            part[S::OOFF + h * D + i] = O;
        }
    }
    if (n_chunks == 1) return;

    // ---- split-K merge by the last CTA of this (sequence, kv head) ------------
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        int *ticket = p.tickets + sq.ticket * p.Hk + g;
        const int prev = atomicAdd(ticket, 1);
        s_flag = (prev == n_chunks - 1);
        if (s_flag) *ticket = 0; // ready for the next launch
    }
    __syncthreads();
    if (!s_flag) return;
    __threadfence();
    const float *part0 = p.part + ((int64_t)sq.chunk0 * p.Hk + g) * S::PF;
    const int64_t cstride = (int64_t)p.Hk * S::PF;
    float *cm = wm;                         // [n_chunks][R] maxima, then weights
    float *cl = wm + n_chunks * R;          // [n_chunks][R] sums
    // (the host keeps n_chunks <= MERGE_CAP)
    for (int idx = tid; idx < n_chunks * R; idx += NT) {
        const int c = idx / R, h = idx % R;
        cm[idx] = __ldcg(part0 + c * cstride + h);
        cl[idx] = __ldcg(part0 + c * cstride + R + h);
    }
    __syncthreads();
    if (tid < r_act) {
        float M = -INFINITY;
        for (int c = 0; c < n_chunks; ++c) M = fmaxf(M, cm[c * R + tid]);
        float L = 0.f;
        for (int c = 0; c < n_chunks; ++c) L += (M == -INFINITY) ? 0.f : cl[c * R + tid] * exp2f(cm[c * R + tid] - M);
        s_M[tid] = M;
        s_L[tid] = L;
    }
    __syncthreads();
    for (int idx = tid; idx < n_chunks * R; idx += NT) {
        const int h = idx % R;
        cm[idx] = (h < r_act && s_M[h] != -INFINITY) ? exp2f(cm[idx] - s_M[h]) : 0.f;
    }
    __syncthreads();
    // every thread owns 4 consecutive outputs; chunks are read 16 at a time
    // with independent loads so the L2 round trips overlap
    const int ncol = r_act * (D / 4);
    for (int col = tid; col < ncol; col += NT) {
        const int h = col / (D / 4), i4 = col % (D / 4);
        const float *src = part0 + S::OOFF + h * D + 4 * i4;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c0 = 0; c0 < n_chunks; c0 += 16) {
            float4 v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u)
                v[u] = (c0 + u < n_chunks) ? __ldcg(reinterpret_cast<const float4 *>(src + (c0 + u) * cstride))
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const float w = (c0 + u < n_chunks) ? cm[(c0 + u) * R + h] : 0.f;
                O.x += w * v[u].x;
                O.y += w * v[u].y;
                O.z += w * v[u].z;
                O.w += w * v[u].w;
            }
        }
        const float L = s_L[h];
        float *dst = outp + h * D + 4 * i4;
        dst[0] = (L > 0.f) ? O.x / L : 0.f;
        dst[1] = (L > 0.f) ? O.y / L : 0.f;
        dst[2] = (L > 0.f) ? O.z / L : 0.f;
        dst[3] = (L > 0.f) ? O.w / L : 0.f;
    }
}

template <int TYPE, int D, int R>
cudaError_t launch_t(const AttnParams &p, const CUtensorMap *tmk, const CUtensorMap *tmv, cudaStream_t st) {
    using S = Shape<TYPE, D, R>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(attn_kernel<TYPE, D, R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             S::SMEM);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.total_chunks, p.Hk);
    cfg.blockDim = dim3(S::W * 32);
    cfg.dynamicSmemBytes = S::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_kernel<TYPE, D, R>, p, *tmk, *tmv);
}

template <int TYPE, int D>
cudaError_t launch_d(const AttnParams &p, const CUtensorMap *tmk, const CUtensorMap *tmv, cudaStream_t st) {
    if (p.r <= 4) return launch_t<TYPE, D, 4>(p, tmk, tmv, st);
    if (p.r == 5) return launch_t<TYPE, D, 5>(p, tmk, tmv, st);
    if (p.r <= 8) return launch_t<TYPE, D, 8>(p, tmk, tmv, st);
    return cudaErrorInvalidValue;
}

template <int TYPE, int D, int R>
int occupancy() {
    using S = Shape<TYPE, D, R>;
    int n = 0;
    cudaFuncSetAttribute(attn_kernel<TYPE, D, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_kernel<TYPE, D, R>, S::W * 32, S::SMEM) !=
        cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    return n > 0 ? n : 1;
}

template <int TYPE, int D>
int occupancy_d(int r) {
    if (r <= 4) return occupancy<TYPE, D, 4>();
    if (r == 5) return occupancy<TYPE, D, 5>();
    return occupancy<TYPE, D, 8>();
}

template <int TYPE, int D>
int merge_cap_d(int r) {
    if (r <= 4) return Shape<TYPE, D, 4>::MERGE_CAP;
    if (r == 5) return Shape<TYPE, D, 5>::MERGE_CAP;
    return Shape<TYPE, D, 8>::MERGE_CAP;
}

} // namespace

size_t attn_partial_floats(int r, int D) {
    const int R = r <= 4 ? 4 : (r == 5 ? 5 : 8);
    return (size_t)(((2 * R + 3) / 4) * 4 + R * D);
}

int attn_ctas_per_sm(int type, int D, int r) {
    if (type == KVC_Q8_0) return D == 128 ? occupancy_d<KVC_Q8_0, 128>(r) : occupancy_d<KVC_Q8_0, 64>(r);
    return D == 128 ? occupancy_d<KVC_F16, 128>(r) : occupancy_d<KVC_F16, 64>(r);
}

int attn_merge_cap(int type, int D, int r) {
    if (type == KVC_Q8_0) return D == 128 ? merge_cap_d<KVC_Q8_0, 128>(r) : merge_cap_d<KVC_Q8_0, 64>(r);
    return D == 128 ? merge_cap_d<KVC_F16, 128>(r) : merge_cap_d<KVC_F16, 64>(r);
}

cudaError_t launch_attn(int type, const AttnParams &p, const CUtensorMap *tmk, const CUtensorMap *tmv,
                        cudaStream_t st) {
    if (type == KVC_Q8_0) {
        if (p.D == 128) return launch_d<KVC_Q8_0, 128>(p, tmk, tmv, st);
        if (p.D == 64) return launch_d<KVC_Q8_0, 64>(p, tmk, tmv, st);
    } else {
        if (p.D == 128) return launch_d<KVC_F16, 128>(p, tmk, tmv, st);
        if (p.D == 64) return launch_d<KVC_F16, 64>(p, tmk, tmv, st);
    }
    return cudaErrorInvalidValue;
}

bool encode_rows_map(CUtensorMap *m, const void *base, int64_t rows, int row_bytes, int type, bool swizzle,
                     std::string *why) {
    using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static EncodeFn fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !ptr) {
            if (why) *why = "cuTensorMapEncodeTiled entry point not found";
            return false;
        }
        fn = reinterpret_cast<EncodeFn>(ptr);
    }
    const bool q8 = type == KVC_Q8_0;
    const int esize = q8 ? 1 : 2;
    const cuuint64_t elems = (cuuint64_t)(row_bytes / esize);
    cuuint64_t gdim[2] = {elems, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)row_bytes};
    // swizzled K: inner box of 128 bytes (or the whole 64-byte row); plain V: the whole row
    cuuint32_t inner = swizzle ? (cuuint32_t)((row_bytes >= 128 ? 128 : row_bytes) / esize) : (cuuint32_t)elems;
    cuuint32_t box[2] = {inner, (cuuint32_t)TMA_BOX_ROWS};
    cuuint32_t estr[2] = {1, 1};
    CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
    if (swizzle) sw = (inner * esize == 128) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    CUresult r = fn(m, q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(base),
                    gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        if (why) *why = "cuTensorMapEncodeTiled failed with code " + std::to_string((int)r);
        return false;
    }
    return true;
}

} // namespace kvc
