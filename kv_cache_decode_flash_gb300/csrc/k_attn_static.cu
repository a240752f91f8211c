// k_attn_static.cu - decode attention over caller-owned K/V buffers that
// allocates nothing.
//
// Some callers cannot let a library call cudaMalloc: serving runtimes that
// reserve all device memory up front and hand it out from their own arena
// (a library-side allocation would break their accounting or fail outright),
// and latency-critical paths where an allocation's implicit device
// synchronisation is not acceptable.  For them this entry point runs the
// same split-K decode attention kernel as kvc_attn_decode, but takes the K/V
// of one sequence directly from caller buffers and keeps the kernel's work
// space (split-K partials, arrival tickets, error word) in one file-scope
// device array of fixed size, so neither this call nor its set-up allocates.
#include "kvc_internal.h"

#include <algorithm>
#include <cstring>

namespace kvc {
namespace {

// Work space shared by every call on a device: tickets, error word, a
// one-entry page table, then the split-K partials.  Every GPU that loads
// the library holds it until the process exits.
constexpr size_t STATIC_SCRATCH_BYTES = 8u << 20;
constexpr size_t TICKET_BYTES = (size_t)MAX_SEQ_PER_LAUNCH * 64 * sizeof(int32_t); // up to 64 KV heads
constexpr size_t HEADER_BYTES = 32768;                                             // tickets + err + page table
static_assert(TICKET_BYTES + 256 <= HEADER_BYTES, "header too small");

static __device__ __align__(256) unsigned char g_attn_scratch[STATIC_SCRATCH_BYTES];

// Per device: the context the entries below belong to, the array's device
// address in that context and the SM count.
uint64_t g_ctx[MAX_DEVICES];
unsigned char *g_scratch_dev[MAX_DEVICES];
int g_sms[MAX_DEVICES];

// First call on a device (and again in a new context of it, e.g. after a
// reset): resolve the array's device address, with the device current (the
// host-side name is only a stand-in for it), and the SM count.
int setup(int dev) {
    const uint64_t ctx = current_context_id();
    if (ctx != 0 && g_ctx[dev] == ctx && g_scratch_dev[dev]) return KVC_OK;
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_attn_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();
        return KVC_ECUDA;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KVC_ECUDA;
    g_sms[dev] = sms;
    g_scratch_dev[dev] = (unsigned char *)ptr;
    g_ctx[dev] = ctx;
    return KVC_OK;
}

} // namespace
} // namespace kvc

extern "C" int kvc_attn_decode_static(int type, int n_head, int n_head_kv, int head_dim, int n_kv, const void *k,
                                      const uint16_t *ks, const void *v, const uint16_t *vs, const float *q,
                                      float *out, float kq_scale, void *stream) {
    using namespace kvc;
    if (type != KVC_Q8_0 && type != KVC_F16) return KVC_EINVAL;
    if (n_head < 1 || n_head_kv < 1 || n_head_kv > 64 || n_head % n_head_kv) return KVC_EINVAL;
    const int r = n_head / n_head_kv;
    if (r > MAX_GROUP || (head_dim != 64 && head_dim != 128) || n_kv < 0) return KVC_EINVAL;
    if (!q || !out || q == out || (n_kv > 0 && (!k || !v))) return KVC_EINVAL;
    if (type == KVC_Q8_0 && n_kv > 0 && (!ks || !vs)) return KVC_EINVAL;
    if (((uintptr_t)q | (uintptr_t)out | (uintptr_t)k | (uintptr_t)v | (uintptr_t)ks | (uintptr_t)vs) & 15)
        return KVC_EINVAL;
    if ((int64_t)n_head_kv * std::max(n_kv, 1) > INT32_MAX) return KVC_ERANGE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return KVC_ECUDA;
    int rc = setup(dev);
    if (rc) return rc;
    unsigned char *base = g_scratch_dev[dev];
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    // split-K plan (one CTA per SM): whole waves of CTAs, 64..ATTN_MAX_CHUNK_ROWS rows per chunk.
    // Occupancy, merge capacity and partial size are those of the instance that runs: plain
    // int8 q8_0 codes run the group-size-8 instance for every group size.
    const int ri = attn_instance_r(type, r, /*raw_codes=*/true);
    const int occ = attn_ctas_per_sm(type, head_dim, ri, 0);
    int64_t slots = (int64_t)g_sms[dev] * occ;
    const int64_t work = std::max<int64_t>((int64_t)n_kv * n_head_kv, 1);
    // short chunks: leave the SMs of a previous launch's last (merging) CTAs free, as the
    // context planner does
    if (occ == 1 && (int64_t)n_head_kv * 8 <= slots && work <= (slots - n_head_kv) * 4096) slots -= n_head_kv;
    const int64_t cmax = ATTN_MAX_CHUNK_ROWS;
    const int64_t waves = std::max<int64_t>(1, (work + slots * cmax - 1) / (slots * cmax));
    int64_t C = (work + waves * slots - 1) / (waves * slots);
    C = std::min<int64_t>(cmax, std::max<int64_t>(64, (C + 15) / 16 * 16));
    const int cap = attn_merge_cap(type, head_dim, ri, 0);
    if ((n_kv + cap - 1) / cap > C) C = ((n_kv + cap - 1) / cap + 15) / 16 * 16;
    C = std::min<int64_t>(C, cmax);
    const int n_chunks = std::max<int>(1, (int)((n_kv + C - 1) / C));
    const size_t part_bytes = (size_t)n_chunks * n_head_kv * attn_partial_floats(ri, head_dim) * sizeof(float);
    if (part_bytes > STATIC_SCRATCH_BYTES - HEADER_BYTES) return KVC_ERANGE; // beyond the fixed work space

    const int row_bytes = type == KVC_Q8_0 ? head_dim : 2 * head_dim;
    const int64_t rows = (int64_t)n_head_kv * std::max(n_kv, 1);
    CUtensorMap tmk[2], tmv[2]; // 16-row and 128-row boxes
    // an empty sequence still needs valid maps; they are never used
    const void *kb = n_kv > 0 ? k : (const void *)(base + HEADER_BYTES);
    const void *vb = n_kv > 0 ? v : (const void *)(base + HEADER_BYTES);
    for (int b = 0; b < 2; ++b) {
        const int box = b ? (int)std::min<int64_t>(TMA_BIG_ROWS, rows) : TMA_BOX_ROWS;
        if (!encode_rows_map(&tmk[b], kb, rows, row_bytes, type, true, nullptr, box) ||
            !encode_rows_map(&tmv[b], vb, rows, row_bytes, type, true, nullptr, box))
            return KVC_ECUDA;
    }

    // tickets, the error word and the one-entry page table (page 0) must start
    // at zero; the array keeps the previous call's contents, so clear them in
    // stream order
    if (cudaMemsetAsync(base, 0, TICKET_BYTES + 32, st) != cudaSuccess) return KVC_ECUDA;

    AttnParams p;
    std::memset(&p, 0, sizeof(p));
    p.H = n_head;
    p.Hk = n_head_kv;
    p.D = head_dim;
    p.r = r;
    p.P = std::max(n_kv, 1);
    p.chunk_rows = (int)C;
    p.n_seq = 1;
    p.total_chunks = n_chunks;
    p.kq_scale_log2 = (float)((double)kq_scale * 1.4426950408889634);
    p.q = q;
    p.out = out;
    p.ks = ks;
    p.vs = vs;
    p.part = reinterpret_cast<float *>(base + HEADER_BYTES);
    p.tickets = reinterpret_cast<int32_t *>(base);
    p.err = reinterpret_cast<uint32_t *>(base + TICKET_BYTES);
    // scale rows are read in 16-byte pieces: the buffers must be readable up to
    // the next multiple of 16 bytes
    const int sb = type == KVC_Q8_0 ? (head_dim / QK) * 2 : 0;
    p.scale_limit_bytes = ((int64_t)n_head_kv * n_kv * sb + 15) / 16 * 16;
    p.map_rows = (int64_t)n_head_kv * std::max(n_kv, 1);
    p.part_cap = (int64_t)((STATIC_SCRATCH_BYTES - HEADER_BYTES) / sizeof(float));
    AttnSeq &a = p.seq[0];
    a.page_table = reinterpret_cast<const int32_t *>(base + TICKET_BYTES + 16);
    a.off = 0;
    a.n_rows = n_kv;
    a.chunk0 = 0;
    a.n_chunks = n_chunks;
    a.out_row = 0;
    a.ticket = 0;
    a.stable_rows = 0; // caller buffers: nothing is read before the dependency wait
    a.pt_len = 1;
    return launch_attn(type, type, p, tmk, tmv, st, /*raw_codes=*/true) == cudaSuccess ? KVC_OK : KVC_ECUDA;
}
