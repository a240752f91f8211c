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
// tiles of 128 rows (never across a page) through a multi-stage shared-memory
// ring filled by one lane of a load warp with TMA: K and V rows as 2-D boxes
// of 128 (and 16) rows, swizzled so that the tensor-core fragment loads are
// bank-conflict free, and the q8_0 scales as 1-D bulk copies.  Tiles of rows
// no in-flight kernel writes are requested before the programmatic-dependency
// wait, so a launch prefetches under the end of the previous one.  The compute
// warps form groups that take tiles in turn; a warp owns one or two 16-row
// slabs of each tile its group takes (two: their products interleave) and runs
// its own online softmax:
//   QK  on the tensor cores (mma.sync m16n8k16, fp32 accumulate): int8 codes
//       become exact fp16 values in registers, q is split into fp16 hi + lo
//       parts (about 22 significant bits), and each 32-element block gets its
//       own accumulator so the block scale is applied in fp32 afterwards;
//   PV  on the tensor cores as O^T = V^T (P' hi + lo)^T, the q8_0 V scale
//       folded into the probability (P' = p * d_v * 2^S per block, with a
//       per-warp range exponent S that keeps hi and lo normal fp16); P' is
//       formed in the accumulator layout of the scores and transposed into
//       the B operand by movmatrix.
// Warps merge inside the CTA; CTAs of one (sequence, kv head) merge through
// global partials, the last CTA to arrive (an atomic ticket, no waiting)
// combining them in fixed chunk order, so results are bitwise repeatable.
// A decode step may also hand the kernel each sequence's new K/V row: the
// CTA whose chunk holds it quantises and stores it before reading its tile.
// Configuration 0 runs one CTA per SM (q8_0: 12 compute warps in 3 groups of
// 4, two slabs each; f16: 8 warps in one group, one slab each); configuration
// 1 (q8_0) two CTAs of 8 compute warps (one slab each) per SM.
#include "kvc_internal.h"
#include "quant_row.cuh"

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
// Bounded wait: gives up after WAIT_LIMIT polls (reported in *err, and *abort
// set so that the CTA's other waits give up too), or as soon as *abort is set.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity, uint32_t *err, volatile int *abort) {
    for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
    }
    atomicOr(err, ERR_WAIT_TIMEOUT);
    *abort = 1;
    return false;
}
// Bounded wait for copies already issued (the drain before a CTA reuses or
// gives back its shared memory): no early exit.
__device__ __forceinline__ bool mbar_wait_landed(uint64_t *bar, unsigned parity, uint32_t *err) {
    for (uint32_t i = 0; i < WAIT_LIMIT; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    atomicOr(err, ERR_WAIT_TIMEOUT);
    return false;
}

// Tile copies carry an L2 policy: the KV stream is read once per step, so its
// lines go first when L2 needs room and the small data around it (queries,
// partials, page tables, the new rows) stays resident.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar,
                                            uint64_t pol) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
                 "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void bulk_load(void *dst, const void *src, unsigned bytes, uint64_t *bar, uint64_t pol) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
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

// Four codes -> two half2 of their exact values: (c0,c1) and (c2,c3).  The
// offset-binary bytes u = c + 128 go into the low mantissa byte of 0x64xx
// (= 1024 + u); subtracting 1152 gives c exactly.  RAW: the word holds plain
// int8 codes, flipped to offset binary first.
template <bool RAW>
__device__ __forceinline__ void codes_to_half2(uint32_t w, uint32_t &h01, uint32_t &h23) {
    const uint32_t u = RAW ? (w ^ CODE_FLIP) : w;
    asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(h01) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(h23) : "r"(u), "r"(0x64646464u));
    const uint32_t bias = 0x64806480u; // half2(1152, 1152)
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(h01) : "r"(bias));
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(h23) : "r"(bias));
}







__device__ __forceinline__ void ldsm_x4(const void *p, uint32_t &a, uint32_t &b, uint32_t &c, uint32_t &d) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_trans(const void *p, uint32_t &a, uint32_t &b, uint32_t &c, uint32_t &d) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "r"(smem_u32(p)));
}
// 2^x (approximate, relative error ~2^-22; +0 for -inf)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Split two fp32 values into fp16 hi + lo pairs: hi keeps the top 11
// significant bits (exactly representable), lo = x - hi rounded to fp16.
__device__ __forceinline__ void split_pack(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const float h0 = __uint_as_float(__float_as_uint(x0) & 0xFFFFE000u);
    const float h1 = __uint_as_float(__float_as_uint(x1) & 0xFFFFE000u);
    const __half2 hh = __floats2half2_rn(h0, h1), ll = __floats2half2_rn(x0 - h0, x1 - h1);
    hi = *reinterpret_cast<const uint32_t *>(&hh);
    lo = *reinterpret_cast<const uint32_t *>(&ll);
}
// Transpose of an 8x8 matrix of halves held as m16n8 accumulator rows (lane
// i: row i/4, columns 2(i%4), 2(i%4)+1) into the same layout of the transpose.
__device__ __forceinline__ uint32_t movt(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
// A transposed V word holds codes (row 2t, dim 2g), (row 2t, dim 2g+1),
// (row 2t+1, dim 2g), (row 2t+1, dim 2g+1); return the exact half2 of the
// even dim (rows 2t, 2t+1) and of the odd dim.
template <bool RAW>
__device__ __forceinline__ void vcodes_to_half2(uint32_t w, uint32_t &ev, uint32_t &od) {
    const uint32_t u = RAW ? (w ^ CODE_FLIP) : w;
    asm("prmt.b32 %0, %1, %2, 0x5240;" : "=r"(ev) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x5341;" : "=r"(od) : "r"(u), "r"(0x64646464u));
    const uint32_t bias = 0x64806480u; // half2(1152, 1152)
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(ev) : "r"(bias));
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(od) : "r"(bias));
}

__device__ __forceinline__ void ldsm_x2_trans(const void *p, uint32_t &a, uint32_t &b) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
                 : "=r"(a), "=r"(b)
                 : "r"(smem_u32(p)));
}
// A transposed word of packed q4_0 bytes holds bytes (row 2t: 2g, 2g+1) and
// (row 2t+1: 2g, 2g+1) of a block, i.e. the codes of dims 2g, 2g+16 (byte 2g)
// and 2g+1, 2g+17 (byte 2g+1) on both rows.  Return the exact half2 (rows 2t,
// 2t+1) of code - 8 for each dim: a nibble or 16 x a nibble goes into the low
// mantissa bits of 1024 (0x6400), then 1032 is subtracted, or the value is
// scaled by 1/16 and 72 subtracted, both exactly.
__device__ __forceinline__ void nibbles_to_half2(uint32_t w, uint32_t &d_lo_e, uint32_t &d_hi_e, uint32_t &d_lo_o,
                                                 uint32_t &d_hi_o) {
    const uint32_t w8 = w >> 8;
    d_lo_e = (w & 0x000F000Fu) | 0x64006400u;  // dim 2g
    d_hi_e = (w & 0x00F000F0u) | 0x64006400u;  // dim 2g + 16
    d_lo_o = (w8 & 0x000F000Fu) | 0x64006400u; // dim 2g + 1
    d_hi_o = (w8 & 0x00F000F0u) | 0x64006400u; // dim 2g + 17
    const uint32_t b1032 = 0x64086408u;          // half2(1032, 1032)
    const uint32_t s16 = 0x2C002C00u, m72 = 0xD480D480u; // half2(1/16), half2(-72)
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(d_lo_e) : "r"(b1032));
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(d_lo_o) : "r"(b1032));
    asm("fma.rn.f16x2 %0, %0, %1, %2;" : "+r"(d_hi_e) : "r"(s16), "r"(m72));
    asm("fma.rn.f16x2 %0, %0, %1, %2;" : "+r"(d_hi_o) : "r"(s16), "r"(m72));
}

// The NB fp16 scales of one row (NB = 2 or 4), one 4- or 8-byte load.
template <int NB>
__device__ __forceinline__ void load_scales(const uint8_t *p, uint32_t (&w)[NB / 2]) {
    if constexpr (NB == 4) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        w[0] = v.x;
        w[1] = v.y;
    } else {
        w[0] = *reinterpret_cast<const uint32_t *>(p);
    }
}
template <int N>
__device__ __forceinline__ float half_at(const uint32_t (&w)[N], int b) {
    return __half2float(__ushort_as_half((uint16_t)(w[b >> 1] >> (16 * (b & 1)))));
}

// 2^e for e in [-126, 127] (exact, from the exponent bits).
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }
// floor(log2 x) of a positive normal float (its unbiased exponent).
__device__ __forceinline__ int ilogb_normal(float x) { return ((__float_as_int(x) >> 23) & 0xff) - 127; }

// Slack of the lazily raised softmax maximum (log2 units): probabilities stay
// below 2^RESCALE_SLACK between raises.
constexpr int RESCALE_SLACK = 8;

// Programmatic dependent launch: wait for the preceding kernel's results /
// let the next kernel be scheduled.  No-ops without a programmatic edge.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Static shape of one kernel instance.  W compute warps in groups of GW;
// group j takes tiles j, j + G, j + 2G, ... and each of its warps owns SL
// slabs of 16 rows of a tile, whose products it interleaves.  One more warp
// issues the tile loads.
template <int TYPE, int D, int R, int CFG = 0, bool V4 = false>
struct Shape {
    static constexpr bool Q8 = TYPE == KVC_Q8_0;
    static_assert(!V4 || (Q8 && D == 128 && CFG == 0), "q4_0 V: with q8_0 K, head_dim 128, configuration 0");
    // CFG 0: one CTA per SM (q8_0: 12 compute warps in 3 groups, two 16-row
    // slabs each); CFG 1 (q8_0): two CTAs per SM of 8 compute warps, each with
    // half the SM's shared memory, for launches whose work exceeds one wave of
    // CFG 0 at the longest chunks
    static constexpr bool FAT = Q8 && CFG == 0;
    static constexpr int SL = FAT ? 2 : 1;            // 16-row slabs per warp and tile
    static constexpr int W = FAT ? 12 : 8;            // compute warps per CTA
    static constexpr int GW = FAT ? 4 : 8;            // warps per group
    static constexpr int G = W / GW;                  // groups
    static constexpr int NTHREADS = (W + 1) * 32;     // compute warps + the load warp
    static constexpr int T = 16 * SL * GW;            // rows per tile
    static constexpr int NB = D / 32;                 // q8_0 blocks per row
    static constexpr int KROW = Q8 ? D : 2 * D;       // bytes per K row
    static constexpr int VROW = V4 ? D / 2 : KROW;    // bytes per V row (q4_0: packed codes)
    static constexpr int SB = Q8 ? NB * 2 : 0;        // scale bytes per row
    static constexpr int KSUB = Q8 ? 1 : (D == 128 ? 2 : 1); // f16 K sub-tiles of 64 halves
    // scale copies start on the 16-byte boundary at or below a tile's first scale row: up to
    // 16 bytes more than the tile's rows hold
    static constexpr int SCALE_BUF = Q8 ? T * SB + 16 : 0;
    static constexpr int KBYTES = T * KROW, VBYTES = T * VROW;
    // K and V tiles of one stage; the swizzled boxes need 1024-byte aligned destinations.
    // The scales of all stages sit after all the tiles.
    static constexpr int STAGE = KBYTES + VBYTES;
    static_assert(STAGE % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
    static constexpr int KSTEPS = D / 16;
    static constexpr int NBX = Q8 ? NB : 1;           // scale blocks per row (1 for f16)
    static constexpr int MAXT = 512;                  // tiles per chunk (host keeps chunks within it)
    static constexpr int QF_BYTES = KSTEPS * 32 * 16 + 64; // q fragments (one copy for all warps) + head scales
    static constexpr int SM_BUDGET = CFG == 1 ? 115712 : 232448; // shared memory one CTA may take
    static constexpr int MINB = CFG == 1 ? 2 : 1;                 // CTAs per SM the registers allow for
    // shared memory besides the stages: base alignment, tile tables, q fragments, and a
    // margin for the kernel's static shared variables
    static constexpr int FIXED = 1024 + MAXT * 8 + 16 + QF_BYTES + 64;
    static constexpr int PER_STAGE = STAGE + 2 * SCALE_BUF + 3 * 8; // tiles, scales, full/empty, tile info
    // as many stages (2..8) as fit, a whole number per group: group j takes tiles
    // j, j + G, ..., so with STAGES a multiple of G every phase of a stage belongs to
    // one group, whose warps consumed the stage's previous tile before waiting on it
    static constexpr int FIT = (SM_BUDGET - FIXED) / PER_STAGE;
    static constexpr int FIT_C = FIT > 8 ? 8 : FIT;
    static constexpr int FIT_G = FIT_C - FIT_C % G;
    static constexpr int STAGES = FIT_G < 2 ? 2 : FIT_G;
    static_assert(STAGES % G == 0, "a stage's phases must all belong to one group");
    static constexpr int OOFF = ((2 * R + 3) / 4) * 4;  // partial: m[R], l[R], pad, then o[R][D] 16-byte aligned
    static constexpr int PF = OOFF + R * D;            // floats of one partial
    static constexpr int SMEM = FIXED + STAGES * PER_STAGE;
    static_assert(SMEM <= SM_BUDGET, "shared memory");
    static constexpr int RING = STAGES * (STAGE + 2 * SCALE_BUF); // tiles + scales, contiguous
    static constexpr int MERGE_CAP = RING / (4 * (PF + R)); // chunks one merge round stages
    // chunks per (sequence, kv head) the planner may use: CFG 0 merges in one
    // round; CFG 1 has little staging room and merges in rounds
    static constexpr int CHUNK_CAP = CFG == 1 ? 256 : MERGE_CAP;
    static constexpr int BIG = 128;                    // rows of a large TMA box (small boxes are 16 rows)
    static constexpr int NMT = D / 16;                 // PV m-tiles of 16 dims
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

// BATCH: every sequence has its own chunk length (AttnSeq.chunk_rows); the
// other instances read the launch's one (AttnParams.chunk_rows).
template <int TYPE, int D, int R, bool RAW = false, int CFG = 0, bool V4 = false, bool BATCH = false>
__global__ void __launch_bounds__(Shape<TYPE, D, R, CFG, V4>::NTHREADS, Shape<TYPE, D, R, CFG, V4>::MINB)
    attn_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmk,
                const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmkb,
                const __grid_constant__ CUtensorMap tmvb) {
    using S = Shape<TYPE, D, R, CFG, V4>;
    constexpr int W = S::W, T = S::T, NT = S::NTHREADS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *stages = smem;                                  // [STAGES][K tile, V tile]
    uint8_t *scales = smem + S::STAGES * S::STAGE;           // [STAGES][K scales, V scales]
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::RING);
    uint64_t *empty = full + S::STAGES;
    TileInfo *tinfo = reinterpret_cast<TileInfo *>(empty + S::STAGES);
    int *s_tstart = reinterpret_cast<int *>(tinfo + S::STAGES); // first row of every tile
    int *s_tpage = s_tstart + S::MAXT;                        // its physical page
    // q fragments of every k-step, lane-major: {hi b0, hi b1, lo b0, lo b1}
    uint4 *qfs = reinterpret_cast<uint4 *>(((uintptr_t)(s_tpage + S::MAXT) + 15) & ~(uintptr_t)15);
    float *shs = reinterpret_cast<float *>(qfs + S::KSTEPS * 32); // 2^-e of each head slot
    __shared__ int s_flag;
    __shared__ int s_nstable; // leading tiles made only of stable rows
    // set by a wait that gave up: the load lane stops issuing and every other wait gives up too
    __shared__ int s_abort;

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
    const int crows = BATCH ? sq.chunk_rows : p.chunk_rows;
    const int row_begin = lc * crows;
    const int row_end = min(sq.n_rows, row_begin + crows);
    // fused quantise-on-append: this CTA's chunk holds the row it stores before reading it
    const bool app = p.app_k != nullptr && sq.app_row >= row_begin && sq.app_row < row_end;

    // tiles never cross a page: their sizes follow from (off, rows, P) alone
    auto tile_rows = [&](int r0) { return min(min(T, row_end - r0), p.P - (sq.off + r0) % p.P); };
    if (tid == 0) {
        int nt = 0, ns = 0;
        for (int r0 = row_begin; r0 < row_end && nt < S::MAXT; r0 += tile_rows(r0)) {
            s_tstart[nt++] = r0;
            if (r0 + tile_rows(r0) <= sq.stable_rows) ns = nt;
        }
        s_flag = nt;
        s_nstable = ns;
        s_abort = 0;
        for (int s = 0; s < S::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], S::GW); // the group of warps that reads the stage
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if constexpr (S::Q8) {
        // Scale bytes past a tile's rows are never copied into: start them at 0
        // (finite), so those rows' products stay 0 without masking
        for (int i = tid; i < S::STAGES * (2 * S::SCALE_BUF / 16); i += NT)
            reinterpret_cast<uint4 *>(scales)[i] = make_uint4(0, 0, 0, 0);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); // before the bulk copies write there
    }
    __syncthreads();
    const int n_tiles = s_flag;
    const int n_stable = s_nstable;
    // Physical page of tile k.  A page outside the page table or the tensor
    // maps is reported and replaced by page 0 (inside every map: the tile reads
    // valid memory, the result is flagged).
    auto tile_page = [&](int k) {
        const int idx = (sq.off + s_tstart[k]) / p.P;
        int page = idx < sq.pt_len ? sq.page_table[idx] : -1;
        if (page < 0 || ((int64_t)page * p.Hk + p.Hk) * p.P > p.map_rows) {
            atomicOr(p.err, ERR_BAD_PAGE);
            page = 0;
        }
        return page;
    };
    // Page-table entries of stable tiles were written by kernels that completed
    // before the preceding launch passed its wait; the others (a page a preceding
    // kernel may just have added) are read after this launch's wait, below.
    if (warp == 0)
        for (int k = lane; k < n_stable; k += 32) s_tpage[k] = tile_page(k);
    __syncthreads();

    // ---- tile loads, all issued by lane 0 of the load warp (warp W) -----------
    const uint64_t pol = l2_evict_first_policy();
    auto issue = [&](int k) {
        const int s = k % S::STAGES;
        const int r0 = s_tstart[k];
        const int n = tile_rows(r0);
        const int page = s_tpage[k];
        const int cell = (sq.off + r0) % p.P;
        const int64_t R0 = ((int64_t)page * p.Hk + g) * p.P + cell;
        uint8_t *st = stages + s * S::STAGE;
        // large boxes first, then 16-row boxes for the rest of the tile
        const int nbig = n / S::BIG;
        const int nsmall = (n - nbig * S::BIG + TMA_BOX_ROWS - 1) / TMA_BOX_ROWS;
        unsigned bytes = (unsigned)((nbig * S::BIG + nsmall * TMA_BOX_ROWS) * (S::KROW + S::VROW));
        int delta = 0;
        unsigned sbytes = 0;
        int64_t saligned = 0;
        if constexpr (S::Q8) {
            const int64_t start = R0 * S::SB;
            saligned = start & ~(int64_t)15;
            delta = (int)((start - saligned) / S::SB);
            const int64_t end = (start + (int64_t)n * S::SB + 15) & ~(int64_t)15;
            sbytes = (unsigned)(end - saligned);
            if (saligned < 0 || saligned + (int64_t)sbytes > p.scale_limit_bytes) {
                atomicOr(p.err, ERR_BAD_INDEX);
                sbytes = 0;
            }
            bytes += 2 * sbytes;
        }
        tinfo[s].n = n;
        tinfo[s].delta = delta;
        mbar_expect_tx(&full[s], bytes);
        auto box = [&](const CUtensorMap *mk, const CUtensorMap *mv, int ro) {
            const int y = (int)(R0 + ro);
            if constexpr (S::KSUB == 1) {
                // rows of at most 128 bytes: one swizzled box per tensor
                tma_load_2d(st + ro * S::KROW, mk, 0, y, &full[s], pol);
                tma_load_2d(st + S::KBYTES + ro * S::VROW, mv, 0, y, &full[s], pol);
            } else {
                // 256-byte f16 rows: two 128-byte sub-tiles per tensor
                tma_load_2d(st + ro * 128, mk, 0, y, &full[s], pol);
                tma_load_2d(st + T * 128 + ro * 128, mk, 64, y, &full[s], pol);
                tma_load_2d(st + S::KBYTES + ro * 128, mv, 0, y, &full[s], pol);
                tma_load_2d(st + S::KBYTES + T * 128 + ro * 128, mv, 64, y, &full[s], pol);
            }
        };
        for (int b = 0; b < nbig; ++b) box(&tmkb, &tmvb, b * S::BIG);
        for (int b = 0; b < nsmall; ++b) box(&tmk, &tmv, nbig * S::BIG + b * TMA_BOX_ROWS);
        if constexpr (S::Q8) {
            if (sbytes) {
                uint8_t *sc = scales + s * (2 * S::SCALE_BUF);
                bulk_load(sc, reinterpret_cast<const uint8_t *>(p.ks) + saligned, sbytes, &full[s], pol);
                bulk_load(sc + S::SCALE_BUF, reinterpret_cast<const uint8_t *>(p.vs) + saligned, sbytes, &full[s], pol);
            }
        }
    };
    // Tiles made only of rows no in-flight kernel writes (the stable prefix)
    // are requested before waiting for the preceding kernel.
    const bool loader = warp == W && lane == 0;
    // Warm L2 with this head group's query rows.  They are read only after the
    // wait below (a preceding kernel may write them); L2 is coherent, so a line
    // brought in early is simply updated by such a write.
    if (warp == 0 && lane < r_act * (D * 4 / 128)) {
        const char *qb = reinterpret_cast<const char *>(p.q + ((int64_t)sq.out_row * p.H + (int64_t)g * r_act) * D);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(qb + lane * 128));
    }
    int prod_k = 0; // tiles issued so far (by the load lane)
    // Before the wait: q8_0 one tile per group (the first round), f16 two tiles of its
    // three; the other stages are requested once the query fragments are built, so that
    // the query's load after the wait does not queue behind the whole prefetch.  (The
    // two-CTA configuration keeps its two stages requested before the wait.)
    constexpr int PRE = S::FAT ? S::G : (S::Q8 ? S::STAGES : 2);
    if (loader)
        while (prod_k < n_stable && prod_k < PRE) issue(prod_k++);
    pdl_wait();
    if (warp == W) {
        // pages of the tiles past the stable prefix, now that preceding kernels are complete
        for (int k = n_stable + lane; k < n_tiles; k += 32) s_tpage[k] = tile_page(k);
        __syncwarp();
        if (lane == 0 && PRE >= S::STAGES) {
            // (the tile of a fused append's row waits until the row is stored)
            for (; prod_k < n_tiles && prod_k < S::STAGES; ++prod_k) {
                if (app && s_tstart[prod_k] + tile_rows(s_tstart[prod_k]) > sq.app_row) break;
                issue(prod_k);
            }
        }
    }

    // per-warp results of the compute warps (read by the CTA merge)
    constexpr int NMT = D / 16;
    float acc[NMT][4];
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[mt][j] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    int sexp = 0;        // P' range exponent S of this warp (valid once have_s)
    bool have_s = false;
    const int gq = lane >> 2, tq = lane & 3;
    // ---- query fragments (B operand of QK), hi + lo fp16.  Warp 0 reads the
    // head group's rows (scaled by kq_scale log2 e) and their maxima, and leaves
    // the values where the fragments go; after a barrier warp ks converts
    // k-step ks in place (each lane its own 16 bytes).
    static_assert(S::KSTEPS <= W, "one converting warp per k-step");
    float4 *qraw = reinterpret_cast<float4 *>(qfs); // [KSTEPS][32 lanes]
    int *s_eq = reinterpret_cast<int *>(shs + 8);        // e of each head slot
    if (warp == 0) {
        const bool hq = gq < r_act; // head slot this lane feeds into the MMA B operand
        const float *qrow = p.q + ((int64_t)sq.out_row * p.H + (int64_t)g * r_act + (hq ? gq : 0)) * D;
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
            float2 x0 = hq ? *reinterpret_cast<const float2 *>(qrow + d0) : make_float2(0.f, 0.f);
            float2 x1 = hq ? *reinterpret_cast<const float2 *>(qrow + d1) : make_float2(0.f, 0.f);
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
#pragma unroll
        for (int ks = 0; ks < S::KSTEPS; ++ks) qraw[ks * 32 + lane] = make_float4(qv[ks][0], qv[ks][1], qv[ks][2], qv[ks][3]);
        if (tq == 0) {
            shs[gq] = ldexpf(1.0f, -e_q);
            s_eq[gq] = e_q;
        }
    }
    if (app && warp == 1) {
        // the new row of KV head g, quantised by the same steps (and to the same bytes) as the
        // append kernel; its cell comes from the page table like every tile's
        const int64_t lr = (int64_t)sq.off + sq.app_row;
        const int64_t idx = lr / p.P;
        const int page = idx < sq.pt_len ? sq.page_table[idx] : -1;
        if (page < 0 || ((int64_t)page * p.Hk + p.Hk) * p.P > p.map_rows) {
            if (lane == 0) atomicOr(p.err, ERR_BAD_PAGE);
        } else {
            const int64_t R = ((int64_t)page * p.Hk + g) * p.P + lr % p.P;
            const int64_t in = ((int64_t)sq.out_row * p.app_heads + g) * D;
            float xk[D / 32], xv[D / 32];
            load_row<D / 32>(p.app_k + in, lane, xk);
            load_row<D / 32>(p.app_v + in, lane, xv);
            store_row<D>(TYPE, p.app_lv.k, R, lane, xk);
            store_row<D>(V4 ? KVC_Q4_0 : TYPE, p.app_lv.v, R, lane, xv);
            // order the stores before the bulk copies (async proxy) issued after the barrier
            asm volatile("fence.proxy.async.global;" ::: "memory");
        }
    }
    __syncthreads();
    if (warp < S::KSTEPS) {
        const int ks = warp;
        const float4 x = qraw[ks * 32 + lane];
        const int e_q = s_eq[gq];
        const float xs[4] = {x.x, x.y, x.z, x.w};
        uint32_t bh[2], bl[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float x0 = ldexpf(xs[2 * j], e_q), x1 = ldexpf(xs[2 * j + 1], e_q);
            const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
            const __half l0 = __float2half_rn(x0 - __half2float(h0)), l1 = __float2half_rn(x1 - __half2float(h1));
            bh[j] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
            bl[j] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
        }
        qfs[ks * 32 + lane] = make_uint4(bh[0], bh[1], bl[0], bl[1]);
    }
    __syncthreads();

    if (warp == W) {
        // the load warp: refill each stage as soon as its group has released it
        if (lane == 0) {
            for (; prod_k < n_tiles && prod_k < S::STAGES; ++prod_k) issue(prod_k);
            for (; prod_k < n_tiles; ++prod_k) {
                const int s = prod_k % S::STAGES;
                if (!mbar_wait(&empty[s], ((prod_k / S::STAGES) - 1) & 1, p.err, &s_abort)) break;
                issue(prod_k);
            }
            // Drain: the last tile issued into each stage has landed before the
            // CTA reuses its shared memory (or exits), also when a wait gave up.
            // The stage's earlier tiles were consumed before that tile was issued,
            // so its full barrier is at most one phase behind and the parity is exact.
            for (int k = max(prod_k - S::STAGES, 0); k < prod_k; ++k)
                mbar_wait_landed(&full[k % S::STAGES], (k / S::STAGES) & 1, p.err);
        }
    } else {

    // 2^-e for the two heads (2t, 2t+1) whose scores this lane accumulates
    const float hs0 = shs[2 * tq], hs1 = shs[2 * tq + 1];

    // ---- per-warp state -------------------------------------------------------
    // softmax state of heads 2t, 2t+1; PV accumulators O^T[dims][heads] as
    // m16n8 fragments (rows = dims, columns = heads 2t, 2t+1)
    constexpr int SL = S::SL;
    const int rbase = (warp % S::GW) * (16 * SL); // this warp's first row in a tile of its group

    for (int k = warp / S::GW; k < n_tiles; k += S::G) {
        const int s = k % S::STAGES;
        if (!mbar_wait(&full[s], (k / S::STAGES) & 1, p.err, &s_abort)) break;
        const uint8_t *st = stages + s * S::STAGE;
        const uint8_t *vt = st + S::KBYTES;
        const uint8_t *sct = scales + s * (2 * S::SCALE_BUF); // K scales, then V scales
        const int n = tinfo[s].n;
        const int rows_w = min(max(n - rbase, 0), 16 * SL);
        // A warp with rows computes all its slabs: a slab past the tile's rows reads
        // stage bytes of an earlier tile (or never written), which are finite for the
        // q8_0 instances (int8 codes, scales zeroed at the start), and its rows are
        // masked to p = 0.  Branching around such a slab costs the interleaving of
        // the two slabs' instructions.  (f16 instances keep one slab per warp.)
        if (rows_w > 0) {
            // ---------------- QK on the tensor cores, slab by slab interleaved ----------------
            // sc[sl]: (row g, 2t) (row g, 2t+1) (row g+8, 2t) (row g+8, 2t+1) of slab sl
            float sc[SL][4];
#pragma unroll
            for (int sl = 0; sl < SL; ++sl) sc[sl][0] = sc[sl][1] = sc[sl][2] = sc[sl][3] = 0.f;
            // ldmatrix lane roles: rows 0-7 / 8-15 of a slab, first / second 16-byte chunk
            const int lm_row = rbase + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int lm_hi = lane >> 4;
            if constexpr (S::Q8) {
                // K scales of rows g, g + 8 of every slab: NB halves each, one 8- (or 4-) byte load per row
                const uint8_t *ksb = sct + (tinfo[s].delta + rbase) * S::SB;
                uint32_t kw[SL][2][S::NB / 2];
#pragma unroll
                for (int sl = 0; sl < SL; ++sl) {
                    load_scales<S::NB>(ksb + (16 * sl + gq) * S::SB, kw[sl][0]);
                    load_scales<S::NB>(ksb + (16 * sl + gq + 8) * S::SB, kw[sl][1]);
                }
#pragma unroll
                for (int b = 0; b < S::NB; ++b) {
                    const uint4 qa = qfs[(2 * b) * 32 + lane], qb = qfs[(2 * b + 1) * 32 + lane];
#pragma unroll
                    for (int sl = 0; sl < SL; ++sl) {
                        uint32_t r0, r1, r2, r3;
                        ldsm_x4(st + swz<S::KROW>(lm_row + 16 * sl, 2 * b + lm_hi), r0, r1, r2, r3);
                        float c[4] = {0.f, 0.f, 0.f, 0.f};
                        uint32_t a0, a1, a2, a3;
                        codes_to_half2<RAW>(r0, a0, a2);
                        codes_to_half2<RAW>(r1, a1, a3);
                        mma16816(c, a0, a1, a2, a3, qa.x, qa.y);
                        mma16816(c, a0, a1, a2, a3, qa.z, qa.w);
                        codes_to_half2<RAW>(r2, a0, a2);
                        codes_to_half2<RAW>(r3, a1, a3);
                        mma16816(c, a0, a1, a2, a3, qb.x, qb.y);
                        mma16816(c, a0, a1, a2, a3, qb.z, qb.w);
                        const float da = half_at(kw[sl][0], b), db = half_at(kw[sl][1], b);
                        sc[sl][0] = fmaf(da, c[0], sc[sl][0]);
                        sc[sl][1] = fmaf(da, c[1], sc[sl][1]);
                        sc[sl][2] = fmaf(db, c[2], sc[sl][2]);
                        sc[sl][3] = fmaf(db, c[3], sc[sl][3]);
                    }
                }
            } else {
                const int lrow = rbase + (lane & 15);
#pragma unroll
                for (int ks = 0; ks < S::KSTEPS; ++ks) {
                    const uint4 qk = qfs[ks * 32 + lane];
#pragma unroll
                    for (int sl = 0; sl < SL; ++sl) {
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4(st + (ks / 4) * T * 128 + swz<128>(lrow + 16 * sl, 2 * (ks % 4) + (lane >> 4)), a0, a1,
                                a2, a3);
                        mma16816(sc[sl], a0, a1, a2, a3, qk.x, qk.y);
                        mma16816(sc[sl], a0, a1, a2, a3, qk.z, qk.w);
                    }
                }
            }
            // log2-domain scores; rows beyond the tile are -inf
            float s2v[SL][4];
#pragma unroll
            for (int sl = 0; sl < SL; ++sl) {
                const int r0 = 16 * sl + gq;
                s2v[sl][0] = (r0 < rows_w) ? sc[sl][0] * hs0 : -INFINITY;
                s2v[sl][1] = (r0 < rows_w) ? sc[sl][1] * hs1 : -INFINITY;
                s2v[sl][2] = (r0 + 8 < rows_w) ? sc[sl][2] * hs0 : -INFINITY;
                s2v[sl][3] = (r0 + 8 < rows_w) ? sc[sl][3] * hs1 : -INFINITY;
            }
            // ---------------- online softmax (per warp) ----------------
            // The running maxima m0, m1 (warp-uniform) are only raised when a
            // score exceeds them by more than RESCALE_SLACK (log2 units), so
            // most tiles need no cross-lane reduction; probabilities are then
            // at most 2^RESCALE_SLACK, which the P' range exponent allows for.
            float t0 = fmaxf(s2v[0][0], s2v[0][2]), t1 = fmaxf(s2v[0][1], s2v[0][3]);
#pragma unroll
            for (int sl = 1; sl < SL; ++sl) {
                t0 = fmaxf(t0, fmaxf(s2v[sl][0], s2v[sl][2]));
                t1 = fmaxf(t1, fmaxf(s2v[sl][1], s2v[sl][3]));
            }
            const bool raise = __any_sync(0xffffffffu, t0 > m0 + RESCALE_SLACK || t1 > m1 + RESCALE_SLACK);
            float mn0 = m0, mn1 = m1;
            if (raise) {
#pragma unroll
                for (int m = 4; m < 32; m <<= 1) {
                    t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, m));
                    t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, m));
                }
                mn0 = fmaxf(m0, t0); // finite: the slabs have a live row
                mn1 = fmaxf(m1, t1);
            }
            // (head slots past the group have q = 0 and feed only columns that are never read)
            float pr[SL][4];
#pragma unroll
            for (int sl = 0; sl < SL; ++sl) {
                pr[sl][0] = ex2(s2v[sl][0] - mn0);
                pr[sl][1] = ex2(s2v[sl][1] - mn1);
                pr[sl][2] = ex2(s2v[sl][2] - mn0);
                pr[sl][3] = ex2(s2v[sl][3] - mn1);
            }
            // ---------------- V scales of the rows this lane holds (g, g + 8 of each slab) -------
            uint32_t vw[SL][2][S::NBX / 2 > 0 ? S::NBX / 2 : 1];
            int s_tile = 14 - RESCALE_SLACK; // f16: P' = p <= 2^RESCALE_SLACK
            if constexpr (S::Q8) {
                const uint8_t *vsb = sct + S::SCALE_BUF + (tinfo[s].delta + rbase) * S::SB;
                uint32_t wm = 0;
#pragma unroll
                for (int sl = 0; sl < SL; ++sl)
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        // rows past the tile hold finite stale scales (or 0): their p is 0, and
                        // the range exponent may only come out smaller than needed (safe)
                        load_scales<S::NB>(vsb + (16 * sl + gq + 8 * i) * S::SB, vw[sl][i]);
#pragma unroll
                        for (int h = 0; h < S::NB / 2; ++h) wm = __vmaxu2(wm, vw[sl][i][h]); // fp16 >= 0: integer order
                    }
                wm = __vmaxu2(wm, __shfl_xor_sync(0xffffffffu, wm, 4));
                wm = __vmaxu2(wm, __shfl_xor_sync(0xffffffffu, wm, 8));
                wm = __vmaxu2(wm, __shfl_xor_sync(0xffffffffu, wm, 16));
                const float dmax = __half2float(__ushort_as_half((uint16_t)max(wm & 0xffffu, wm >> 16)));
                // 2^S * max(p * d) < 2^15 with p <= 2^RESCALE_SLACK: hi and lo of P' stay in fp16 range
                // dmax is an fp16 value: a normal float in [2^-24, 2^16), so S stays in [-9, 30]
                s_tile = (dmax > 0.f) ? 14 - RESCALE_SLACK - ilogb_normal(dmax) : (have_s ? sexp : 0);
            }
            const int s_new = have_s ? min(sexp, s_tile) : s_tile;
            // rescale the accumulators: the softmax maxima moved and/or S decreased
            if (raise || s_new != sexp || !have_s) {
                const float sf = have_s ? pow2i(s_new - sexp) : 1.f;
                const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1); // 0 while m is -inf
                const float f0 = al0 * sf, f1 = al1 * sf;
#pragma unroll
                for (int mt = 0; mt < NMT; ++mt) {
                    acc[mt][0] *= f0;
                    acc[mt][1] *= f1;
                    acc[mt][2] *= f0;
                    acc[mt][3] *= f1;
                }
                l0 *= f0;
                l1 *= f1;
                m0 = mn0;
                m1 = mn1;
            }
            // per-lane partial row sums, in the same 2^S domain as the accumulators
            const float ps = pow2i(s_new);
#pragma unroll
            for (int sl = 0; sl < SL; ++sl) {
                l0 = fmaf(pr[sl][0] + pr[sl][2], ps, l0);
                l1 = fmaf(pr[sl][1] + pr[sl][3], ps, l1);
                pr[sl][0] *= ps;
                pr[sl][1] *= ps;
                pr[sl][2] *= ps;
                pr[sl][3] *= ps;
            }
            sexp = s_new;
            have_s = true;
            // ---------------- PV on the tensor cores: O^T += V^T (P' hi + lo)^T --------------
            // P' of a slab sits as accumulator rows (row g | g + 8, heads 2t, 2t+1); its hi and
            // lo halves, transposed by movmatrix, are the B fragments (rows 2t, 2t+1 | 2t+8,
            // 2t+9 of head g).
#pragma unroll
            for (int b = 0; b < S::NBX; ++b) {
#pragma unroll
                for (int sl = 0; sl < SL; ++sl) {
                    float x[4];
                    if constexpr (S::Q8) {
                        const float dg = half_at(vw[sl][0], b), dg8 = half_at(vw[sl][1], b);
                        x[0] = pr[sl][0] * dg;
                        x[1] = pr[sl][1] * dg;
                        x[2] = pr[sl][2] * dg8;
                        x[3] = pr[sl][3] * dg8;
                    } else {
                        x[0] = pr[sl][0]; // rows past the tile have p = 0
                        x[1] = pr[sl][1];
                        x[2] = pr[sl][2];
                        x[3] = pr[sl][3];
                    }
                    uint32_t hg, lg, hg8, lg8;
                    split_pack(x[0], x[1], hg, lg);
                    split_pack(x[2], x[3], hg8, lg8);
                    const uint32_t b0h = movt(hg), b1h = movt(hg8), b0l = movt(lg), b1l = movt(lg8);
                    const int vrow = lm_row + 16 * sl;
                    if constexpr (V4) {
                        // block b is one 16-byte chunk of each 64-byte row: ra = rows 0-7,
                        // rb = rows 8-15; nibble pairs give the same even / odd dim
                        // m-tiles as the int8 codes (dims 2g | 2g+16 and 2g+1 | 2g+17)
                        uint32_t ra, rb;
                        ldsm_x2_trans(vt + swz<S::VROW>(vrow, b), ra, rb);
                        uint32_t e0, e1, e2, e3, o0, o1, o2, o3;
                        nibbles_to_half2(ra, e0, e1, o0, o1);
                        nibbles_to_half2(rb, e2, e3, o2, o3);
                        mma16816(acc[2 * b], e0, e1, e2, e3, b0h, b1h);
                        mma16816(acc[2 * b], e0, e1, e2, e3, b0l, b1l);
                        mma16816(acc[2 * b + 1], o0, o1, o2, o3, b0h, b1h);
                        mma16816(acc[2 * b + 1], o0, o1, o2, o3, b0l, b1l);
                    } else if constexpr (S::Q8) {
                        uint32_t v0, v1, v2, v3;
                        ldsm_x4_trans(vt + swz<S::VROW>(vrow, 2 * b + lm_hi), v0, v1, v2, v3);
                        // v0: rows 0-7 / bytes 0-15, v1: rows 8-15 / bytes 0-15,
                        // v2: rows 0-7 / bytes 16-31, v3: rows 8-15 / bytes 16-31 of block b
                        uint32_t e0, e1, e2, e3, o0, o1, o2, o3;
                        vcodes_to_half2<RAW>(v0, e0, o0);
                        vcodes_to_half2<RAW>(v2, e1, o1);
                        vcodes_to_half2<RAW>(v1, e2, o2);
                        vcodes_to_half2<RAW>(v3, e3, o3);
                        mma16816(acc[2 * b], e0, e1, e2, e3, b0h, b1h);
                        mma16816(acc[2 * b], e0, e1, e2, e3, b0l, b1l);
                        mma16816(acc[2 * b + 1], o0, o1, o2, o3, b0h, b1h);
                        mma16816(acc[2 * b + 1], o0, o1, o2, o3, b0l, b1l);
                    } else {
                        // f16: the single "block" spans all D dims, NMT m-tiles of 16 dims
                        const int lv_row = rbase + 16 * sl + (lane & 7) + (lane >> 4) * 8;
                        const int lv_c = (lane >> 3) & 1;
#pragma unroll
                        for (int mt = 0; mt < NMT; ++mt) {
                            uint32_t a0, a1, a2, a3;
                            ldsm_x4_trans(vt + (mt / 4) * T * 128 + swz<128>(lv_row, 2 * (mt % 4) + lv_c), a0, a1,
                                          a2, a3);
                            mma16816(acc[mt], a0, a1, a2, a3, b0h, b1h);
                            mma16816(acc[mt], a0, a1, a2, a3, b0l, b1l);
                        }
                    }
                }
            }
        }
        // release the stage; the last warp done with it loads tile k + STAGES into it
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]); // release: this warp's reads of the stage are complete
    }
    } // compute warps
    __syncthreads();
    // the next launch may be scheduled now (it waits for this grid's end before reading);
    // its CTAs land on SMs as this launch's CTAs leave
    pdl_trigger();

    // ---- CTA merge of the warps (stages are free now) -------------------------
    // Each warp stores its fragments as they sit in registers (lane-major,
    // conflict free), its softmax state and its P' range exponent.
    constexpr int FRAG = S::NMT * 32;                           // float4 fragments per warp
    float4 *wf = reinterpret_cast<float4 *>(stages);           // [W][NMT][32]
    float *wm = reinterpret_cast<float *>(wf + W * FRAG);      // [W][8]
    float *wl = wm + W * 8;                                     // [W][8]
    float *wus = wl + W * 8;                                    // [W]
    float *wwt = wus + W;                                       // [W][8] merge weights
    float *wmx = wwt + W * 8;                                   // [8] the CTA's maxima
    if (warp < W) {
#pragma unroll
        for (int mt = 0; mt < S::NMT; ++mt)
            wf[(warp * S::NMT + mt) * 32 + lane] = make_float4(acc[mt][0], acc[mt][1], acc[mt][2], acc[mt][3]);
        // row sums: lanes gq = 0..7 hold different rows of the same heads
#pragma unroll
        for (int m = 4; m < 32; m <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, m);
            l1 += __shfl_xor_sync(0xffffffffu, l1, m);
        }
        if (gq == 0) {
            wm[warp * 8 + 2 * tq] = m0;
            wm[warp * 8 + 2 * tq + 1] = m1;
            wl[warp * 8 + 2 * tq] = l0;
            wl[warp * 8 + 2 * tq + 1] = l1;
        }
        if (lane == 0) wus[warp] = have_s ? pow2i(-sexp) : 0.f;
    }
    __syncthreads();
    // the weight of warp w in head slot h: 2^(m_w - M) * 2^-S_w (0 for a warp without rows)
    if (tid < W * 8) {
        const int h = tid & 7;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < W; ++w) M = fmaxf(M, wm[w * 8 + h]);
        wwt[tid] = (M == -INFINITY) ? 0.f : ex2(wm[tid] - M) * wus[tid >> 3];
        if (tid < 8) wmx[h] = M;
    }
    __syncthreads();

    const int n_chunks = sq.n_chunks;
    float *part = p.part + ((int64_t)(sq.part0 + lc) * p.Hk + g) * S::PF;
    const bool part_ok = ((int64_t)(sq.part0 + lc) * p.Hk + g + 1) * S::PF <= p.part_cap;
    if (!part_ok && tid == 0 && n_chunks > 1) atomicOr(p.err, ERR_BAD_PART);
    float *outp = p.out + ((int64_t)sq.out_row * p.H + (int64_t)g * r_act) * D;
    // fragment (mt, ln): heads 2t, 2t+1 of lane ln, dims of rows g and g+8: the
    // warps' fragments summed with those weights (softmax rescale and the warp's
    // 2^-S: O and l of a warp share its 2^S domain), in warp order.
    for (int it = tid; it < FRAG; it += NT) {
        const int mt = it / 32, ln = it % 32, fg = ln >> 2, ft = ln & 3;
        const int h0 = 2 * ft, h1 = 2 * ft + 1;
        const float M0 = wmx[h0], M1 = wmx[h1];
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        float L0 = 0.f, L1 = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            const float2 f = *reinterpret_cast<const float2 *>(wwt + w * 8 + h0); // h0 even: (h0, h1)
            const float f0 = f.x, f1 = f.y;
            const float4 v = wf[(w * S::NMT + mt) * 32 + ln];
            O.x = fmaf(f0, v.x, O.x);
            O.y = fmaf(f1, v.y, O.y);
            O.z = fmaf(f0, v.z, O.z);
            O.w = fmaf(f1, v.w, O.w);
            L0 = fmaf(f0, wl[w * 8 + h0], L0);
            L1 = fmaf(f1, wl[w * 8 + h1], L1);
        }
        int dA, dB;
        if constexpr (S::Q8) {
            dA = 32 * (mt / 2) + 2 * fg + (mt % 2);
            dB = dA + 16;
        } else {
            dA = 16 * mt + fg;
            dB = dA + 8;
        }
        if (n_chunks == 1) {
            if (h0 < r_act) {
                outp[h0 * D + dA] = (L0 > 0.f) ? O.x / L0 : 0.f;
                outp[h0 * D + dB] = (L0 > 0.f) ? O.z / L0 : 0.f;
            }
            if (h1 < r_act) {
                outp[h1 * D + dA] = (L1 > 0.f) ? O.y / L1 : 0.f;
                outp[h1 * D + dB] = (L1 > 0.f) ? O.w / L1 : 0.f;
            }
        } else if (part_ok) {
            if (h0 < R) {
                part[S::OOFF + h0 * D + dA] = O.x;
                part[S::OOFF + h0 * D + dB] = O.z;
            }
            if (h1 < R) {
                part[S::OOFF + h1 * D + dA] = O.y;
                part[S::OOFF + h1 * D + dB] = O.w;
            }
            if (mt == 0 && fg == 0) { // one writer per head pair: the partial's max and sum
                if (h0 < r_act) {
                    part[h0] = M0;
                    part[R + h0] = L0;
                }
                if (h1 < r_act) {
                    part[h1] = M1;
                    part[R + h1] = L1;
                }
            }
        }
    }
    if (n_chunks == 1) return;

    // ---- split-K merge by the last CTA of this (sequence, kv head) ------------
    __syncthreads();
    if (tid == 0) {
        // release: this CTA's partial (cumulative over the barrier above) is
        // visible before the ticket; the last arrival acquires all of them
        int *ticket = p.tickets + sq.ticket * p.Hk + g;
        int prev;
        asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(prev) : "l"(ticket) : "memory");
        s_flag = (prev == n_chunks - 1);
        if (s_flag) *ticket = 0; // ready for the next launch
    }
    __syncthreads();
    if (!s_flag) return;
    const float *part0 = p.part + ((int64_t)sq.part_first * p.Hk + g) * S::PF;
    const int64_t cstride = (int64_t)p.Hk * S::PF;
    if (((int64_t)(sq.part_first + n_chunks - 1) * p.Hk + g + 1) * S::PF > p.part_cap) {
        // reported above or by the CTA that wrote past the buffer: nothing to merge
        if (tid == 0) atomicOr(p.err, ERR_BAD_PART);
        return;
    }
    // The partials are merged in rounds of at most MERGE_CAP chunks, each
    // staged in shared memory by one round of independent loads.  A thread
    // owns one output column (4 dims of one head) and keeps its running
    // maximum, weight sum and weighted output across rounds, rescaled when a
    // round raises the maximum; within a round the chunks go in chunk order.
    // The same bits on every call; one round gives the plain merge.
    static_assert(8 * (D / 4) <= NT, "one output column per thread");
    constexpr int Q4 = S::PF / 4; // float4 per partial
    float4 *stg = reinterpret_cast<float4 *>(stages);
    const float *sp = reinterpret_cast<const float *>(stg);
    const int col = tid, ncol = r_act * (D / 4);
    const int h = col / (D / 4), i4 = col % (D / 4);
    float Mrun = -INFINITY, L = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < n_chunks; c0 += S::MERGE_CAP) {
        const int nc = min(S::MERGE_CAP, n_chunks - c0);
        if (c0 > 0) __syncthreads(); // the previous round's reads of the staging are done
        const int items = nc * Q4;
        for (int base = 0; base < items; base += 8 * NT) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int it = base + u * NT + tid;
                v[u] = (it < items)
                           ? __ldcg(reinterpret_cast<const float4 *>(part0 + (c0 + it / Q4) * cstride) + it % Q4)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int it = base + u * NT + tid;
                if (it < items) stg[it] = v[u];
            }
        }
        __syncthreads();
        if (col < ncol) {
            float M = -INFINITY;
            for (int c = 0; c < nc; ++c) M = fmaxf(M, sp[c * S::PF + h]);
            if (M != -INFINITY) {
                const float Mn = fmaxf(Mrun, M);
                if (Mrun != -INFINITY && Mn != Mrun) {
                    const float a = ex2(Mrun - Mn);
                    O.x *= a;
                    O.y *= a;
                    O.z *= a;
                    O.w *= a;
                    L *= a;
                }
                for (int c = 0; c < nc; ++c) {
                    const float w = ex2(sp[c * S::PF + h] - Mn);
                    const float4 v = *reinterpret_cast<const float4 *>(sp + c * S::PF + S::OOFF + h * D + 4 * i4);
                    L = fmaf(w, sp[c * S::PF + R + h], L);
                    O.x = fmaf(w, v.x, O.x);
                    O.y = fmaf(w, v.y, O.y);
                    O.z = fmaf(w, v.z, O.z);
                    O.w = fmaf(w, v.w, O.w);
                }
                Mrun = Mn;
            }
        }
    }
    if (col < ncol) {
        float *dst = outp + h * D + 4 * i4;
        dst[0] = (L > 0.f) ? O.x / L : 0.f;
        dst[1] = (L > 0.f) ? O.y / L : 0.f;
        dst[2] = (L > 0.f) ? O.z / L : 0.f;
        dst[3] = (L > 0.f) ? O.w / L : 0.f;
    }
}

template <int TYPE, int D, int R, bool RAW = false, int CFG = 0, bool V4 = false, bool BATCH = false>
cudaError_t launch_t(const AttnParams &p, const CUtensorMap *tmk, const CUtensorMap *tmv, cudaStream_t st) {
    // tmk / tmv point at {16-row map, 128-row map} pairs
    using S = Shape<TYPE, D, R, CFG, V4>;
    // the shared-memory attribute belongs to the current context: set it once per
    // context of each device (a reset device or another context gets it again)
    static uint64_t configured[MAX_DEVICES];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t ctx = current_context_id();
    if (dev < 0 || dev >= MAX_DEVICES || ctx == 0 || configured[dev] != ctx) {
        e = cudaFuncSetAttribute(attn_kernel<TYPE, D, R, RAW, CFG, V4, BATCH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 S::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < MAX_DEVICES) configured[dev] = ctx;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.total_chunks, p.Hk);
    cfg.blockDim = dim3(S::NTHREADS);
    cfg.dynamicSmemBytes = S::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_kernel<TYPE, D, R, RAW, CFG, V4, BATCH>, p, tmk[0], tmv[0], tmk[1], tmv[1]);
}

template <int TYPE, int D>
cudaError_t launch_d(const AttnParams &p, const CUtensorMap *tmk, const CUtensorMap *tmv, cudaStream_t st,
                     bool raw, int cfg, bool v4) {
    if (v4) {
        // q4_0 V: q8_0 K, head_dim 128, configuration 0 only
        if constexpr (TYPE == KVC_Q8_0 && D == 128) {
            if (raw || cfg != 0) return cudaErrorInvalidValue;
            if (p.r <= 4) return launch_t<TYPE, D, 4, false, 0, true>(p, tmk, tmv, st);
            if (p.r == 5) return launch_t<TYPE, D, 5, false, 0, true>(p, tmk, tmv, st);
            if (p.r <= 8) return launch_t<TYPE, D, 8, false, 0, true>(p, tmk, tmv, st);
        }
        return cudaErrorInvalidValue;
    }
    if (p.n_seq > 1) {
        // a batch: per-sequence chunk lengths (symmetric types; plain launch configurations)
        if (raw) return cudaErrorInvalidValue;
        if constexpr (TYPE == KVC_Q8_0) {
            if (cfg == 1) {
                if (p.r <= 4) return launch_t<TYPE, D, 4, false, 1, false, true>(p, tmk, tmv, st);
                if (p.r == 5) return launch_t<TYPE, D, 5, false, 1, false, true>(p, tmk, tmv, st);
                if (p.r <= 8) return launch_t<TYPE, D, 8, false, 1, false, true>(p, tmk, tmv, st);
                return cudaErrorInvalidValue;
            }
        }
        if (p.r <= 4) return launch_t<TYPE, D, 4, false, 0, false, true>(p, tmk, tmv, st);
        if (p.r == 5) return launch_t<TYPE, D, 5, false, 0, false, true>(p, tmk, tmv, st);
        if (p.r <= 8) return launch_t<TYPE, D, 8, false, 0, false, true>(p, tmk, tmv, st);
        return cudaErrorInvalidValue;
    }
    // plain int8 codes (caller buffers): one instance for every group size up to 8
    if constexpr (TYPE == KVC_Q8_0) {
        if (raw) return p.r <= 8 ? launch_t<TYPE, D, 8, true>(p, tmk, tmv, st) : cudaErrorInvalidValue;
        if (cfg == 1) {
            if (p.r <= 4) return launch_t<TYPE, D, 4, false, 1>(p, tmk, tmv, st);
            if (p.r == 5) return launch_t<TYPE, D, 5, false, 1>(p, tmk, tmv, st);
            if (p.r <= 8) return launch_t<TYPE, D, 8, false, 1>(p, tmk, tmv, st);
            return cudaErrorInvalidValue;
        }
    }
    if (p.r <= 4) return launch_t<TYPE, D, 4>(p, tmk, tmv, st);
    if (p.r == 5) return launch_t<TYPE, D, 5>(p, tmk, tmv, st);
    if (p.r <= 8) return launch_t<TYPE, D, 8>(p, tmk, tmv, st);
    return cudaErrorInvalidValue;
}

template <int TYPE, int D, int R, int CFG>
int occupancy() {
    using S = Shape<TYPE, D, R, CFG>;
    int n = 0;
    cudaFuncSetAttribute(attn_kernel<TYPE, D, R, false, CFG>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_kernel<TYPE, D, R, false, CFG>, S::NTHREADS,
                                                      S::SMEM) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    return n > 0 ? n : 1;
}

template <int TYPE, int D, int CFG>
int occupancy_d(int r) {
    if (r <= 4) return occupancy<TYPE, D, 4, CFG>();
    if (r == 5) return occupancy<TYPE, D, 5, CFG>();
    return occupancy<TYPE, D, 8, CFG>();
}

template <int TYPE, int D, int CFG>
int chunk_cap_d(int r) {
    if (r <= 4) return Shape<TYPE, D, 4, CFG>::CHUNK_CAP;
    if (r == 5) return Shape<TYPE, D, 5, CFG>::CHUNK_CAP;
    return Shape<TYPE, D, 8, CFG>::CHUNK_CAP;
}

} // namespace

uint64_t current_context_id() {
    using GetCurrentFn = CUresult (*)(CUcontext *);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long *);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    if (!get_current || !get_id) {
        cudaDriverEntryPointQueryResult q1, q2;
        void *p1 = nullptr, *p2 = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess || !p1 ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &p2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
            q2 != cudaDriverEntryPointSuccess || !p2) {
            cudaGetLastError();
            return 0;
        }
        get_current = reinterpret_cast<GetCurrentFn>(p1);
        get_id = reinterpret_cast<GetIdFn>(p2);
    }
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (get_current(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
    return (uint64_t)id + 1; // 0 stays "unknown"
}

int attn_instance_r(int type, int r, bool raw_codes) {
    if (type == KVC_Q8_0 && raw_codes) return 8; // one instance for every group size
    return r <= 4 ? 4 : (r == 5 ? 5 : 8);
}

size_t attn_partial_floats(int r, int D) {
    const int R = r <= 4 ? 4 : (r == 5 ? 5 : 8);
    return (size_t)(((2 * R + 3) / 4) * 4 + R * D);
}

int attn_ctas_per_sm(int type, int D, int r, int cfg) {
    if (type == KVC_Q8_0) {
        if (cfg == 1) return D == 128 ? occupancy_d<KVC_Q8_0, 128, 1>(r) : occupancy_d<KVC_Q8_0, 64, 1>(r);
        return D == 128 ? occupancy_d<KVC_Q8_0, 128, 0>(r) : occupancy_d<KVC_Q8_0, 64, 0>(r);
    }
    if (cfg == 1) return 0; // f16 has one configuration
    return D == 128 ? occupancy_d<KVC_F16, 128, 0>(r) : occupancy_d<KVC_F16, 64, 0>(r);
}

int attn_merge_cap(int type, int D, int r, int cfg) {
    if (type == KVC_Q8_0) {
        if (cfg == 1) return D == 128 ? chunk_cap_d<KVC_Q8_0, 128, 1>(r) : chunk_cap_d<KVC_Q8_0, 64, 1>(r);
        return D == 128 ? chunk_cap_d<KVC_Q8_0, 128, 0>(r) : chunk_cap_d<KVC_Q8_0, 64, 0>(r);
    }
    return D == 128 ? chunk_cap_d<KVC_F16, 128, 0>(r) : chunk_cap_d<KVC_F16, 64, 0>(r);
}

cudaError_t launch_attn(int type, int type_v, const AttnParams &p, const CUtensorMap *tmk, const CUtensorMap *tmv,
                        cudaStream_t st, bool raw_codes, int cfg) {
    const bool v4 = type_v == KVC_Q4_0;
    if (!v4 && type_v != type) return cudaErrorInvalidValue;
    if (type == KVC_Q8_0) {
        if (p.D == 128) return launch_d<KVC_Q8_0, 128>(p, tmk, tmv, st, raw_codes, cfg, v4);
        if (p.D == 64) return launch_d<KVC_Q8_0, 64>(p, tmk, tmv, st, raw_codes, cfg, v4);
    } else if (!v4) {
        if (cfg != 0) return cudaErrorInvalidValue;
        if (p.D == 128) return launch_d<KVC_F16, 128>(p, tmk, tmv, st, false, 0, false);
        if (p.D == 64) return launch_d<KVC_F16, 64>(p, tmk, tmv, st, false, 0, false);
    }
    return cudaErrorInvalidValue;
}

bool encode_rows_map(CUtensorMap *m, const void *base, int64_t rows, int row_bytes, int type, bool swizzle,
                     std::string *why, int box_rows) {
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
    const bool q8 = type != KVC_F16; // q8_0 codes and packed q4_0 codes: bytes
    const int esize = q8 ? 1 : 2;
    const cuuint64_t elems = (cuuint64_t)(row_bytes / esize);
    cuuint64_t gdim[2] = {elems, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)row_bytes};
    // swizzled K: inner box of 128 bytes (or the whole 64-byte row); plain V: the whole row
    cuuint32_t inner = swizzle ? (cuuint32_t)((row_bytes >= 128 ? 128 : row_bytes) / esize) : (cuuint32_t)elems;
    cuuint32_t box[2] = {inner, (cuuint32_t)box_rows};
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
