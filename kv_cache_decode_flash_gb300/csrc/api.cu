// api.cu - the C ABI (include/kvc.h): validation, the cache manager (host
// metadata of sequences, pages and positions) and the sequence and state
// operations.  The host-resident transport lives in transport.cu.
#include "ctx.h"

#include <cuda_fp16.h>

#include <algorithm>
#include <chrono>
#include <climits>
#include <cmath>
#include <cstring>
#include <new>
#include <thread>

namespace kvc {

// ---------------------------------------------------------------- helpers --

int cuda_fail(Ctx *c, cudaError_t e, const char *what) {
    return c->fail(KVC_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

#define KVC_CU(c, call)                                                                                            \
    do {                                                                                                           \
        cudaError_t e_ = (call);                                                                                   \
        if (e_ != cudaSuccess) return cuda_fail((c), e_, #call);                                                   \
    } while (0)

static bool take_alloc(Ctx *c) {
    if (c->fail_after < 0) return true;
    if (c->fail_after == 0) return false;
    --c->fail_after;
    return true;
}

int dev_alloc(Ctx *c, void **p, int64_t bytes, const char *what) {
    *p = nullptr;
    if (bytes <= 0) return KVC_OK;
    if (!take_alloc(c)) return c->fail(KVC_ENOMEM, std::string("injected allocation failure: ") + what);
    cudaError_t e = cudaMalloc(p, (size_t)bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        return c->fail(KVC_ENOMEM, std::string("cudaMalloc failed for ") + what + ": " + cudaGetErrorString(e));
    }
    c->device_bytes += bytes;
    return KVC_OK;
}

void dev_free(Ctx *c, void *p, int64_t bytes) {
    if (!p) return;
    cudaFree(p);
    c->device_bytes -= bytes;
}

// Wait for the internal stream with a deadline (polling; never an unbounded
// block).  Short waits spin; past 2 ms the poll sleeps between queries.
int wait_internal(Ctx *c) {
    KVC_CU(c, cudaMemcpyAsync(c->err_host, c->err_dev, 4, cudaMemcpyDeviceToHost, c->st));
    KVC_CU(c, cudaEventRecord(c->done, c->st));
    auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        cudaError_t e = cudaEventQuery(c->done);
        if (e == cudaSuccess) break;
        if (e != cudaErrorNotReady) return cuda_fail(c, e, "device work of a synchronous operation");
        auto us = std::chrono::duration_cast<std::chrono::microseconds>(std::chrono::steady_clock::now() - t0).count();
        if (us > (int64_t)c->timeout_ms * 1000) return c->fail(KVC_ETIMEDOUT, "timed out waiting for device work");
        if (us > 2000) std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
    const uint32_t word = *(volatile uint32_t *)c->err_host;
    if (word) return c->fail(KVC_EINTERNAL, "a kernel reported device error word " + std::to_string(word));
    return KVC_OK;
}

// Synchronous operations first wait for all device work issued so far.
int enter_sync(Ctx *c) {
    KVC_CU(c, cudaSetDevice(c->dev));
    KVC_CU(c, cudaDeviceSynchronize());
    c->clear_recent();
    for (uint8_t *p : c->up_retired) cudaFreeHost(p);
    c->up_retired.clear();
    c->up_used = 0;
    return KVC_OK;
}

// Host-to-device copy of a small host array on the internal stream, through
// the pinned upload arena (an asynchronous copy; the caller's array may be
// reused at once).  Falls back to a pageable copy if pinned memory is short.
static int upload(Ctx *c, void *dst, const void *src, int64_t bytes) {
    if (bytes <= 0) return KVC_OK;
    const int64_t need = (bytes + 255) / 256 * 256;
    if (c->up_used + need > c->up_cap) {
        const int64_t cap = std::max<int64_t>({2 * c->up_cap, need, (int64_t)1 << 20});
        uint8_t *p = nullptr;
        if (cudaMallocHost((void **)&p, (size_t)cap) != cudaSuccess) {
            cudaGetLastError();
            KVC_CU(c, cudaMemcpyAsync(dst, src, (size_t)bytes, cudaMemcpyHostToDevice, c->st));
            return KVC_OK;
        }
        if (c->up_host) c->up_retired.push_back(c->up_host);
        c->up_host = p;
        c->up_cap = cap;
        c->up_used = 0;
    }
    uint8_t *h = c->up_host + c->up_used;
    std::memcpy(h, src, (size_t)bytes);
    c->up_used += need;
    KVC_CU(c, cudaMemcpyAsync(dst, h, (size_t)bytes, cudaMemcpyHostToDevice, c->st));
    return KVC_OK;
}

static int ensure_staging(Ctx *c, int64_t bytes) {
    if (bytes <= c->staging_bytes) return KVC_OK;
    dev_free(c, c->staging, c->staging_bytes);
    c->staging = nullptr;
    c->staging_bytes = 0;
    int64_t want = std::max<int64_t>(bytes, 1 << 20);
    int rc = dev_alloc(c, (void **)&c->staging, want, "staging");
    if (rc) return rc;
    c->staging_bytes = want;
    return KVC_OK;
}

// Upload a run list to the device.
static int upload_runs(Ctx *c, const std::vector<RowRun> &runs) {
    if (runs.empty()) return KVC_OK;
    if ((int64_t)runs.size() > c->runs_cap) {
        dev_free(c, c->runs_dev, c->runs_cap * (int64_t)sizeof(RowRun));
        c->runs_dev = nullptr;
        c->runs_cap = 0;
        int64_t cap = std::max<int64_t>((int64_t)runs.size(), 1024);
        int rc = dev_alloc(c, (void **)&c->runs_dev, cap * (int64_t)sizeof(RowRun), "run list");
        if (rc) return rc;
        c->runs_cap = cap;
    }
    return upload(c, c->runs_dev, runs.data(), (int64_t)(runs.size() * sizeof(RowRun)));
}

static int ensure_copy_stream(Ctx *c) {
    if (c->st_copy) return KVC_OK;
    KVC_CU(c, cudaStreamCreateWithFlags(&c->st_copy, cudaStreamNonBlocking));
    for (auto &ev : c->st_ev) KVC_CU(c, cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
    return KVC_OK;
}

// Re-upload the page tables of `s` (synchronous path).
static int upload_pages(Ctx *c, int s) {
    Seq &q = c->seqs[s];
    if (!q.pages.empty()) {
        const int rc = upload(c, c->pt_dev + (int64_t)s * c->max_pages, q.pages.data(), (int64_t)q.pages.size() * 4);
        if (rc) return rc;
    }
    q.dev_pages = (int32_t)q.pages.size();
    return KVC_OK;
}

// Physical row index of (page, kv head, cell) in a layer pool.
static inline int64_t prow(const Ctx *c, int32_t page, int g, int32_t cell) {
    return ((int64_t)page * c->Hk + g) * c->P + cell;
}

static inline void phys(const Ctx *c, const Seq &q, int64_t r, int32_t &page, int32_t &cell) {
    const int64_t lr = r + q.off;
    page = q.pages[(size_t)(lr / c->P)];
    cell = (int32_t)(lr % c->P);
}

// The rows of a sequence whose positions fall in [p0, p1), in row order.
// The usual selection is one contiguous range of rows, which needs no index
// list; the first pass (counts and extremes only) finds out.
struct RowSel {
    int64_t first = 0, count = 0;
    int64_t pos_min = 0, pos_max = -1; // of the selected positions
    bool contiguous = true;            // rows first .. first + count - 1
    std::vector<int64_t> idx;          // the rows, when not contiguous
    int64_t row(int64_t i) const { return contiguous ? first + i : idx[(size_t)i]; }
};

// Pages needed to hold rows [0, n) of a sequence with offset off.
static inline int32_t pages_for(const Ctx *c, int32_t off, int64_t n) {
    return n <= 0 ? 0 : (int32_t)((off + n + c->P - 1) / c->P);
}

// Grow sequence `s` by `add` rows (pages only; positions and counts are the
// caller's).  Returns the indices of the new pages in q.pages via `first_new`.
static int grow_pages(Ctx *c, Seq &q, int64_t add, size_t *first_new) {
    *first_new = q.pages.size();
    const int32_t need = pages_for(c, q.off, (int64_t)q.n + add);
    if (need > c->max_pages) return c->fail(KVC_ENOSPC, "sequence would exceed the page table");
    const int32_t extra = need - (int32_t)q.pages.size();
    if (extra > (int32_t)c->free_pages.size()) return c->fail(KVC_ENOSPC, "no free pages");
    for (int32_t i = 0; i < extra; ++i) {
        q.pages.push_back(c->free_pages.back());
        c->free_pages.pop_back();
    }
    return KVC_OK;
}

static void release_tail_pages(Ctx *c, Seq &q) {
    const int32_t need = pages_for(c, q.off, q.n);
    while ((int32_t)q.pages.size() > need) {
        c->free_pages.push_back(q.pages.back());
        q.pages.pop_back();
    }
    if (q.n == 0) q.off = 0;
    q.dev_pages = std::min<int32_t>(q.dev_pages, (int32_t)q.pages.size());
}

// Pool copy arguments of this context (no payload).
static RunCopyArgs pool_args(const Ctx *c) {
    RunCopyArgs a;
    std::memset(&a, 0, sizeof(a));
    a.base[0] = c->kdata;
    a.base[1] = c->vdata;
    a.base[2] = c->ksb ? c->kscales : nullptr;
    a.base[3] = c->vsb ? c->vscales : nullptr;
    a.rowb[0] = c->krow;
    a.rowb[1] = c->vrow;
    a.rowb[2] = c->ksb;
    a.rowb[3] = c->vsb;
    a.pool_rows = c->pool_rows;
    a.err = c->err_dev;
    return a;
}

// Runs copying logical rows [a, a+len) of sequence qa to logical rows
// [b, b+len) of qb (every layer and tensor: see RowRun).
static void add_row_copies(const Ctx *c, const Seq &qa, int64_t a, const Seq &qb, int64_t b, int64_t len,
                           std::vector<RowRun> &out) {
    int64_t done = 0;
    while (done < len) {
        int32_t pa, ca, pb, cb;
        phys(c, qa, a + done, pa, ca);
        phys(c, qb, b + done, pb, cb);
        int64_t run = std::min<int64_t>(len - done, std::min<int64_t>(c->P - ca, c->P - cb));
        for (int g = 0; g < c->Hk; ++g) out.push_back(RowRun{prow(c, pa, g, ca), prow(c, pb, g, cb), (int32_t)run, 0});
        done += run;
    }
}

static inline int64_t pad16(int64_t x) { return (x + 15) / 16 * 16; }

// State format sizes (see include/kvc.h).
static int64_t section_bytes(const Ctx *c, int type, int64_t n) {
    if (type == KVC_Q8_0) return pad16((int64_t)c->Hk * n * c->D) + pad16((int64_t)c->Hk * n * (c->D / QK) * 2);
    if (type == KVC_Q4_0) return pad16((int64_t)c->Hk * n * (c->D / 2)) + pad16((int64_t)c->Hk * n * (c->D / QK) * 2);
    return pad16((int64_t)c->Hk * n * c->D * 2);
}
static int64_t payload_bytes(const Ctx *c, int64_t n) {
    return (int64_t)c->L * (section_bytes(c, c->tk, n) + section_bytes(c, c->tv, n));
}
static int64_t state_bytes(const Ctx *c, int64_t n) { return 64 + pad16(4 * n) + payload_bytes(c, n); }

// Runs between the pools and a packed payload laid out as in the state
// format, for the rows idx[] of sequence q (row i of the selection is payload
// row g * N + i of head g, N = idx.size()).
static void add_payload_copies(const Ctx *c, const Seq &q, const RowSel &sel, std::vector<RowRun> &out) {
    const int64_t n = sel.count;
    for (int64_t i = 0; i < n;) {
        int32_t pg, cl;
        phys(c, q, sel.row(i), pg, cl);
        int64_t j;
        if (sel.contiguous) {
            j = std::min<int64_t>(n, i + (c->P - cl));
        } else {
            j = i + 1;
            while (j < n && sel.idx[(size_t)j] == sel.idx[(size_t)j - 1] + 1 && cl + (j - i) < c->P) ++j;
        }
        for (int g = 0; g < c->Hk; ++g)
            out.push_back(RowRun{prow(c, pg, g, cl), (int64_t)g * n + i, (int32_t)(j - i), 0});
        i = j;
    }
}
// The contiguous selection of rows [first, first + count).
static RowSel row_range(int64_t first, int64_t count) {
    RowSel s;
    s.first = first;
    s.count = count;
    return s;
}

// Copy arguments between the pools and a payload of n rows per head.
static RunCopyArgs payload_args(const Ctx *c, int64_t n, uint8_t *payload, bool to_payload) {
    RunCopyArgs a = pool_args(c);
    a.payload = payload;
    a.to_payload = to_payload ? 1 : 0;
    // the state format carries plain int8 codes
    a.flip[0] = c->tk == KVC_Q8_0 ? CODE_FLIP : 0u;
    a.flip[1] = c->tv == KVC_Q8_0 ? CODE_FLIP : 0u;
    const int64_t ks = section_bytes(c, c->tk, n);
    a.layer_bytes = ks + section_bytes(c, c->tv, n);
    a.toff[0] = 0;
    a.toff[2] = pad16((int64_t)c->Hk * n * c->krow);
    a.toff[1] = ks;
    a.toff[3] = ks + pad16((int64_t)c->Hk * n * c->vrow);
    a.payload_rows = (int64_t)c->Hk * n;
    return a;
}

// Layer groups of the chunked state copies: group i is layers
// [L i / k, L (i + 1) / k), k = min(L, STATE_CHUNKS).
static inline int state_chunks(const Ctx *c) { return std::min(c->L, Ctx::STATE_CHUNKS); }
static inline int chunk_layer(const Ctx *c, int i) { return (int)((int64_t)c->L * i / state_chunks(c)); }

// Zero the padding bytes of every section of a host payload.
static void zero_payload_pads(const Ctx *c, uint8_t *payload, int64_t n) {
    int64_t off = 0;
    for (int l = 0; l < c->L; ++l)
        for (int t = 0; t < 2; ++t) {
            const int type = t == 0 ? c->tk : c->tv;
            const int64_t db = (int64_t)c->Hk * n * (t == 0 ? c->krow : c->vrow);
            std::memset(payload + off + db, 0, (size_t)(pad16(db) - db));
            if (type != KVC_F16) {
                const int64_t sb = (int64_t)c->Hk * n * (t == 0 ? c->ksb : c->vsb);
                std::memset(payload + off + pad16(db) + sb, 0, (size_t)(pad16(sb) - sb));
            }
            off += section_bytes(c, type, n);
        }
}

// Whether p[0 .. n) are consecutive integers in order.
static bool consecutive(const int32_t *p, int64_t n) {
    if (n <= 1) return true;
    const int64_t p0 = p[0];
    int32_t bad = 0;
    for (int64_t i = 1; i < n; ++i) bad |= p[i] ^ (int32_t)(p0 + i);
    return bad == 0;
}

static void select_rows(const Seq &q, int64_t p0, int64_t p1, RowSel &s) {
    s = RowSel();
    const int64_t lo64 = std::max<int64_t>(p0, 0), hi64 = std::min<int64_t>(p1 - 1, INT32_MAX); // inclusive
    if (q.n <= 0 || hi64 < lo64) return;
    if (q.linear) { // row r holds position pos[0] + r
        const int64_t b0 = q.pos[0];
        const int64_t r0 = std::max<int64_t>(lo64 - b0, 0), r1 = std::min<int64_t>(hi64 - b0, (int64_t)q.n - 1);
        if (r1 < r0) return;
        s.first = r0;
        s.count = r1 - r0 + 1;
        s.pos_min = b0 + r0;
        s.pos_max = b0 + r1;
        return;
    }
    const int32_t lo = (int32_t)lo64, hi = (int32_t)hi64, n = q.n;
    const int32_t *pos = q.pos.data();
    int32_t cnt = 0, r_min = INT32_MAX, r_max = -1, p_min = INT32_MAX, p_max = INT32_MIN;
    for (int32_t r = 0; r < n; ++r) {
        const int32_t p = pos[r];
        const bool in = p >= lo && p <= hi;
        cnt += in ? 1 : 0;
        r_min = std::min(r_min, in ? r : INT32_MAX);
        r_max = std::max(r_max, in ? r : -1);
        p_min = std::min(p_min, in ? p : INT32_MAX);
        p_max = std::max(p_max, in ? p : INT32_MIN);
    }
    if (cnt == 0) return;
    s.first = r_min;
    s.count = cnt;
    s.pos_min = p_min;
    s.pos_max = p_max;
    s.contiguous = (int64_t)r_max - r_min + 1 == cnt;
    if (!s.contiguous) {
        s.idx.reserve((size_t)cnt);
        for (int32_t r = r_min; r <= r_max; ++r)
            if (pos[r] >= lo && pos[r] <= hi) s.idx.push_back(r);
    }
}

static void norm_range(int p0, int p1, int64_t &a, int64_t &b) {
    a = p0 < 0 ? 0 : p0;
    b = p1 < 0 ? (int64_t)INT32_MAX + 1 : p1;
}

} // namespace kvc

using namespace kvc;

// -------------------------------------------------------------- transport --
namespace kvc {
int transport_attn(Ctx *c, int layer, const float *q, float *out, float kq_scale, cudaStream_t st);
int transport_append(Ctx *c, int layer, int n_tok, const float *k, const float *v, int in_heads, cudaStream_t st);
void transport_release(Ctx *c);
int launch_attention(Ctx *c, const LayerView &lv, const CUtensorMap *tmk, const CUtensorMap *tmv, int P,
                     int64_t scale_limit, int n_seq, const AttnSeq *seqs_in, const float *q, float *out,
                     float kq_scale, cudaStream_t st, const float *app_k = nullptr,
                     const float *app_v = nullptr);
} // namespace kvc

// ------------------------------------------------------------------ ABI ----

extern "C" {

void kvc_params_init(kvc_params *p) {
    if (!p) return;
    std::memset(p, 0, sizeof(*p));
    p->n_layer = 1;
    p->n_head = 8;
    p->n_head_kv = 2;
    p->head_dim = 64;
    p->n_ctx = 512;
    p->n_seq_max = 1;
    p->type_k = KVC_Q8_0;
    p->type_v = KVC_Q8_0;
    p->rope_base = 10000.0f;
    p->rope_mode = KVC_ROPE_NEOX;
    p->residency = KVC_DEVICE;
    p->device = 0;
    p->page_rows = 0;
    p->gpu_heads = 0;
}

const char *kvc_status_str(int s) {
    switch (s) {
    case KVC_OK: return "ok";
    case KVC_EINVAL: return "invalid argument";
    case KVC_ENOMEM: return "out of memory";
    case KVC_ENOSPC: return "no space";
    case KVC_ERANGE: return "out of range";
    case KVC_EFORMAT: return "bad state format";
    case KVC_ECUDA: return "CUDA error";
    case KVC_ETIMEDOUT: return "timed out";
    case KVC_EINTERNAL: return "internal error";
    default: return "unknown status";
    }
}

const char *kvc_last_error(const kvc_ctx *c) {
    if (!c) return "null context";
    return reinterpret_cast<const Ctx *>(c)->err.c_str();
}

void kvc_destroy(kvc_ctx *cc) {
    if (!cc) return;
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    if (c->split) {
        kvc_destroy(reinterpret_cast<kvc_ctx *>(c->part_dev));
        kvc_destroy(reinterpret_cast<kvc_ctx *>(c->part_host));
        delete c;
        return;
    }
    cudaSetDevice(c->dev);
    cudaDeviceSynchronize();
    transport_release(c);
    if (c->tr.ordered.kdata) {
        cudaFree(c->tr.ordered.kdata);
        cudaFree(c->tr.ordered.vdata);
        cudaFree(c->tr.ordered.kscales);
        cudaFree(c->tr.ordered.vscales);
    }
    cudaFree(c->kdata);
    cudaFree(c->vdata);
    cudaFree(c->kscales);
    cudaFree(c->vscales);
    cudaFree(c->pt_dev);
    cudaFree(c->part);
    cudaFree(c->tickets);
    cudaFree(c->err_dev);
    if (c->err_host) cudaFreeHost(c->err_host);
    if (c->up_host) cudaFreeHost(c->up_host);
    for (uint8_t *p : c->up_retired) cudaFreeHost(p);
    cudaFree(c->staging);
    cudaFree(c->runs_dev);
    cudaFree(c->spans_dev);
    cudaFree(c->zero_pt);
    if (c->hk) cudaFreeHost(c->hk);
    if (c->hv) cudaFreeHost(c->hv);
    if (c->hks) cudaFreeHost(c->hks);
    if (c->hvs) cudaFreeHost(c->hvs);
    for (auto ev : c->app_ev)
        if (ev) cudaEventDestroy(ev);
    if (c->st) cudaStreamDestroy(c->st);
    if (c->done) cudaEventDestroy(c->done);
    if (c->st_copy) cudaStreamDestroy(c->st_copy);
    for (auto ev : c->st_ev)
        if (ev) cudaEventDestroy(ev);
    for (auto ev : c->trace.pool)
        if (ev) cudaEventDestroy(ev);
    delete c;
}

int kvc_create(const kvc_params *p, kvc_ctx **out) {
    if (!p || !out) return KVC_EINVAL;
    *out = nullptr;
    Ctx *c = new (std::nothrow) Ctx();
    if (!c) return KVC_ENOMEM;
    c->prm = *p;
    auto bad = [&](const char *m) {
        c->err = m;
        delete c;
        return KVC_EINVAL;
    };
    if (p->n_layer < 1 || p->n_head < 1 || p->n_head_kv < 1 || p->n_head % p->n_head_kv) return bad("bad head counts");
    if (p->head_dim != 64 && p->head_dim != 128) return bad("head_dim must be 64 or 128");
    if (p->n_head / p->n_head_kv > MAX_GROUP) return bad("more than 8 query heads per KV head");
    if (p->n_ctx < 1 || p->n_seq_max < 1) return bad("n_ctx and n_seq_max must be positive");
    if ((p->type_k != KVC_Q8_0 && p->type_k != KVC_F16) ||
        (p->type_v != KVC_Q8_0 && p->type_v != KVC_F16 && p->type_v != KVC_Q4_0))
        return bad("type_k must be KVC_Q8_0 or KVC_F16, type_v KVC_Q8_0, KVC_F16 or KVC_Q4_0");
    if (p->type_v == KVC_Q4_0) {
        // the asymmetric cache: q8_0 K, q4_0 V
        if (p->type_k != KVC_Q8_0 || p->head_dim != 128) return bad("q4_0 V needs q8_0 K and head_dim 128");
    } else if (p->type_k != p->type_v) {
        return bad("K and V must have the same type (or q8_0 K with q4_0 V)");
    }
    if (p->rope_mode != KVC_ROPE_NEOX && p->rope_mode != KVC_ROPE_NORM) return bad("bad rope_mode");
    if (!(p->rope_base > 1.0f) || !std::isfinite(p->rope_base)) return bad("rope_base must be > 1");
    if (p->residency != KVC_DEVICE && p->residency != KVC_HOST_PINNED && p->residency != KVC_SPLIT_HEADS)
        return bad("bad residency");
    int page_rows = p->page_rows ? p->page_rows : 256;
    if (page_rows < 16 || page_rows > 4096 || page_rows % 16) return bad("page_rows must be a multiple of 16 in [16, 4096]");
    if (p->residency == KVC_HOST_PINNED && p->n_seq_max != 1) return bad("host-resident contexts hold one sequence");
    if (p->residency == KVC_SPLIT_HEADS) {
        if (p->n_seq_max != 1) return bad("split contexts hold one sequence");
        if (p->gpu_heads < 1 || p->gpu_heads >= p->n_head_kv) return bad("gpu_heads must be in [1, n_head_kv - 1]");
        // two whole contexts on the disjoint KV-head ranges (whole GQA groups)
        const int r = p->n_head / p->n_head_kv;
        kvc_params dp = *p, hp = *p;
        dp.residency = KVC_DEVICE;
        dp.n_head_kv = p->gpu_heads;
        dp.n_head = p->gpu_heads * r;
        hp.residency = KVC_HOST_PINNED;
        hp.n_head_kv = p->n_head_kv - p->gpu_heads;
        hp.n_head = hp.n_head_kv * r;
        kvc_ctx *d = nullptr, *h = nullptr;
        int rc = kvc_create(&dp, &d);
        if (rc == KVC_OK) rc = kvc_create(&hp, &h);
        if (rc != KVC_OK) {
            kvc_destroy(d);
            c->err = "creating a part of the split context failed";
            delete c;
            return rc;
        }
        c->split = true;
        c->host = true; // the sequence and state operations are not available
        c->gpu_heads = p->gpu_heads;
        c->part_dev = reinterpret_cast<Ctx *>(d);
        c->part_host = reinterpret_cast<Ctx *>(h);
        c->dev = p->device;
        c->H = p->n_head;
        c->Hk = p->n_head_kv;
        c->D = p->head_dim;
        c->r = r;
        c->L = p->n_layer;
        c->tk = p->type_k;
        c->tv = p->type_v;
        *out = reinterpret_cast<kvc_ctx *>(c);
        return KVC_OK;
    }

    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || p->device < 0 || p->device >= ndev) {
        cudaGetLastError();
        c->err = "no such CUDA device";
        delete c;
        return KVC_ECUDA;
    }
    c->dev = p->device;
    cudaSetDevice(c->dev);
    cudaDeviceGetAttribute(&c->sms, cudaDevAttrMultiProcessorCount, c->dev);
    c->H = p->n_head;
    c->Hk = p->n_head_kv;
    c->D = p->head_dim;
    c->r = c->H / c->Hk;
    c->L = p->n_layer;
    c->tk = p->type_k;
    c->tv = p->type_v;
    c->krow = c->tk == KVC_Q8_0 ? c->D : 2 * c->D;
    c->vrow = c->tv == KVC_Q8_0 ? c->D : (c->tv == KVC_Q4_0 ? c->D / 2 : 2 * c->D);
    c->ksb = c->tk == KVC_Q8_0 ? (c->D / QK) * 2 : 0;
    c->vsb = c->tv != KVC_F16 ? (c->D / QK) * 2 : 0;
    c->host = p->residency == KVC_HOST_PINNED;
    c->occ = attn_ctas_per_sm(c->tk, c->D, c->r, 0);
    // the two-CTA configuration exists for symmetric q8_0 only
    c->occ2 = c->tv == c->tk ? attn_ctas_per_sm(c->tk, c->D, c->r, 1) : 0;

    auto fail = [&](int rc) {
        kvc_destroy(reinterpret_cast<kvc_ctx *>(c));
        return rc;
    };
    int rc;
    if (cudaStreamCreateWithFlags(&c->st, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&c->done, cudaEventDisableTiming) != cudaSuccess) {
        c->err = "stream/event creation failed";
        return fail(KVC_ECUDA);
    }
    if ((rc = dev_alloc(c, (void **)&c->err_dev, 4, "error word"))) return fail(rc);
    cudaMemsetAsync(c->err_dev, 0, 4, c->st);
    if (cudaMallocHost((void **)&c->err_host, 4) != cudaSuccess) {
        c->err_host = nullptr;
        c->err = "cudaMallocHost failed for the error word";
        return fail(KVC_ENOMEM);
    }
    *c->err_host = 0;
    if ((rc = dev_alloc(c, (void **)&c->tickets, (int64_t)MAX_SEQ_PER_LAUNCH * c->Hk * 4, "tickets")))
        return fail(rc);
    cudaMemsetAsync(c->tickets, 0, (size_t)MAX_SEQ_PER_LAUNCH * c->Hk * 4, c->st);

    if (!c->host) {
        c->P = page_rows;
        c->n_pages = (int32_t)((p->n_ctx + c->P - 1) / c->P) + p->n_seq_max;
        c->max_pages = c->n_pages;
        c->pool_rows = (int64_t)c->n_pages * c->Hk * c->P;
        c->kdata_bytes = (int64_t)c->L * c->pool_rows * c->krow + 64;
        c->vdata_bytes = (int64_t)c->L * c->pool_rows * c->vrow + 64;
        c->kscale_bytes = c->ksb ? (int64_t)c->L * c->pool_rows * c->ksb + 64 : 0;
        c->vscale_bytes = c->vsb ? (int64_t)c->L * c->pool_rows * c->vsb + 64 : 0;
        if ((rc = dev_alloc(c, (void **)&c->kdata, c->kdata_bytes, "K pool"))) return fail(rc);
        if ((rc = dev_alloc(c, (void **)&c->vdata, c->vdata_bytes, "V pool"))) return fail(rc);
        if ((rc = dev_alloc(c, (void **)&c->kscales, c->kscale_bytes, "K scales"))) return fail(rc);
        if ((rc = dev_alloc(c, (void **)&c->vscales, c->vscale_bytes, "V scales"))) return fail(rc);
        // zeroed so that rows never written read as finite zeros
        cudaMemsetAsync(c->kdata, 0, c->kdata_bytes, c->st);
        cudaMemsetAsync(c->vdata, 0, c->vdata_bytes, c->st);
        if (c->kscales) cudaMemsetAsync(c->kscales, 0, c->kscale_bytes, c->st);
        if (c->vscales) cudaMemsetAsync(c->vscales, 0, c->vscale_bytes, c->st);
        if ((rc = dev_alloc(c, (void **)&c->pt_dev, (int64_t)p->n_seq_max * c->max_pages * 4, "page tables")))
            return fail(rc);
        cudaMemsetAsync(c->pt_dev, 0, (size_t)p->n_seq_max * c->max_pages * 4, c->st);
        c->free_pages.reserve(c->n_pages);
        for (int32_t i = c->n_pages - 1; i >= 0; --i) c->free_pages.push_back(i);
        c->tmk.resize(2 * (size_t)c->L);
        c->tmv.resize(2 * (size_t)c->L);
        const int64_t rows_all = (int64_t)c->L * c->pool_rows;
        if (rows_all > INT32_MAX) {
            c->err = "pool too large for 32-bit TMA row coordinates";
            return fail(KVC_EINVAL);
        }
        for (int l = 0; l < c->L; ++l) {
            std::string why;
            for (int b = 0; b < 2; ++b) {
                const int box = b ? (int)std::min<int64_t>(TMA_BIG_ROWS, c->pool_rows) : TMA_BOX_ROWS;
                if (!encode_rows_map(&c->tmk[2 * l + b], c->kdata + (int64_t)l * c->pool_rows * c->krow, c->pool_rows,
                                     c->krow, c->tk, true, &why, box) ||
                    !encode_rows_map(&c->tmv[2 * l + b], c->vdata + (int64_t)l * c->pool_rows * c->vrow, c->pool_rows,
                                     c->vrow, c->tv, true, &why, box)) {
                    c->err = why;
                    return fail(KVC_ECUDA);
                }
            }
        }
        // partials for chunks of at least 64 rows; grown on demand for smaller forced chunks
        const int64_t chunks = (int64_t)p->n_ctx / 64 + 2 * (int64_t)p->n_seq_max + c->sms;
        c->part_floats = chunks * c->Hk * (int64_t)attn_partial_floats(c->r, c->D);
        if ((rc = dev_alloc(c, (void **)&c->part, c->part_floats * 4, "partials"))) return fail(rc);
    } else {
        c->P = p->n_ctx;
        const int64_t rows = (int64_t)c->L * c->Hk * p->n_ctx;
        const int64_t bk = rows * c->krow + 64, bv = rows * c->vrow + 64;
        const int64_t bks = c->ksb ? rows * c->ksb + 64 : 0, bvs = c->vsb ? rows * c->vsb + 64 : 0;
        auto halloc = [&](uint8_t **h, uint8_t **d, int64_t b) -> int {
            if (!b) return KVC_OK;
            if (!take_alloc(c)) return c->fail(KVC_ENOMEM, "injected allocation failure: host store");
            if (cudaHostAlloc((void **)h, (size_t)b, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) {
                cudaGetLastError();
                *h = nullptr;
                return c->fail(KVC_ENOMEM, "cudaHostAlloc failed for the host store");
            }
            std::memset(*h, 0, (size_t)b);
            if (cudaHostGetDevicePointer((void **)d, *h, 0) != cudaSuccess)
                return c->fail(KVC_ECUDA, "cudaHostGetDevicePointer failed");
            c->host_bytes += b;
            return KVC_OK;
        };
        if ((rc = halloc(&c->hk, &c->hk_d, bk)) || (rc = halloc(&c->hv, &c->hv_d, bv)) ||
            (rc = halloc(&c->hks, &c->hks_d, bks)) || (rc = halloc(&c->hvs, &c->hvs_d, bvs)))
            return fail(rc);
        if ((rc = dev_alloc(c, (void **)&c->zero_pt, 4, "slot page table"))) return fail(rc);
        c->app_ev.assign((size_t)c->L, nullptr);
        c->app_gen.assign((size_t)c->L, 0);
        c->tr.app_waited.assign((size_t)c->L, -1);
        for (auto &ev : c->app_ev)
            if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) {
                c->err = "event creation failed";
                return fail(KVC_ECUDA);
            }
        cudaMemsetAsync(c->zero_pt, 0, 4, c->st);
        const int64_t chunks = (int64_t)p->n_ctx / 64 + 2 + c->sms;
        c->part_floats = chunks * c->Hk * (int64_t)attn_partial_floats(c->r, c->D);
        if ((rc = dev_alloc(c, (void **)&c->part, c->part_floats * 4, "partials"))) return fail(rc);
    }
    c->seqs.resize(p->n_seq_max);
    for (auto &q : c->seqs) q.lfill.assign(c->L, 0);
    c->recent.assign(p->n_seq_max, std::vector<int32_t>(c->L, 0));
    if (cudaStreamSynchronize(c->st) != cudaSuccess) {
        c->err = "initialisation failed";
        return fail(KVC_ECUDA);
    }
    *out = reinterpret_cast<kvc_ctx *>(c);
    return KVC_OK;
}

// Append n_tok rows of every KV head of c; k / v hold in_heads head-rows per
// token, of which the first Hk are c's.
static int append_impl(Ctx *c, int layer, int seq, int pos0, int n_tok, const float *k, const float *v,
                       void *stream, int in_heads);

int kvc_append(kvc_ctx *cc, int layer, int seq, int pos0, int n_tok, const float *k, const float *v,
               void *stream) {
    if (!cc) return KVC_EINVAL;
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    if (c->split) {
        if (layer < 0 || layer >= c->L) return c->fail(KVC_EINVAL, "layer out of range");
        if (seq != 0) return c->fail(KVC_EINVAL, "sequence id out of range");
        if (n_tok < 1 || !k || !v) return c->fail(KVC_EINVAL, "n_tok must be >= 1 and k, v non-null");
        if (((uintptr_t)k | (uintptr_t)v) & 15) return c->fail(KVC_EINVAL, "k and v must be 16-byte aligned");
        // the host half first: the host store is the one that can be full (the device half holds the
        // same number of cells in pages); the two halves carry identical positions
        const int64_t skip = (int64_t)c->gpu_heads * c->D;
        int rc = append_impl(c->part_host, layer, seq, pos0, n_tok, k + skip, v + skip, stream, c->Hk);
        if (rc) return c->fail(rc, c->part_host->err);
        rc = append_impl(c->part_dev, layer, seq, pos0, n_tok, k, v, stream, c->Hk);
        if (rc) return c->fail(rc, "device half: " + c->part_dev->err + " (the host half took the rows)");
        return KVC_OK;
    }
    return append_impl(c, layer, seq, pos0, n_tok, k, v, stream, c->Hk);
}

// Checks of an append that change nothing; *creates: the layer is the first to
// append these positions (it allocates the rows).
static int append_check(Ctx *c, int layer, int seq, int pos0, int n_tok, bool *creates) {
    if (layer < 0 || layer >= c->L) return c->fail(KVC_EINVAL, "layer out of range");
    if (seq < 0 || seq >= (int)c->seqs.size()) return c->fail(KVC_EINVAL, "sequence id out of range");
    if (pos0 < 0 || (int64_t)pos0 + n_tok - 1 > INT32_MAX) return c->fail(KVC_ERANGE, "positions out of range");
    const Seq &q = c->seqs[seq];
    const int32_t fill = q.lfill[layer];
    *creates = fill == q.n;
    if (!*creates) {
        if ((int64_t)fill + n_tok > q.n) return c->fail(KVC_EINVAL, "append runs past the rows other layers created");
        for (int i = 0; i < n_tok; ++i)
            if (q.pos[(size_t)fill + i] != pos0 + i)
                return c->fail(KVC_EINVAL, "append positions differ from the rows other layers created");
    }
    return KVC_OK;
}

// Destination of the next n_tok rows of `seq` in `layer` of a device context;
// when the layer creates them, their pages are allocated and new page-table
// entries are sent on st (as kernel arguments, no host copy).
static int device_append_dst(Ctx *c, int layer, int seq, bool creates, int n_tok, cudaStream_t st, AppendDst *d) {
    Seq &q = c->seqs[seq];
    if (creates) {
        size_t first_new;
        int rc = grow_pages(c, q, n_tok, &first_new);
        if (rc) return rc;
        std::vector<int32_t> idx, val;
        for (size_t i = (size_t)q.dev_pages; i < q.pages.size(); ++i) {
            idx.push_back((int32_t)((int64_t)seq * c->max_pages + (int64_t)i));
            val.push_back(q.pages[i]);
        }
        if (!idx.empty()) {
            cudaError_t e = launch_pt_update(c->pt_dev, (int)idx.size(), idx.data(), val.data(), st);
            if (e != cudaSuccess) return cuda_fail(c, e, "page table update");
            q.dev_pages = (int32_t)q.pages.size();
        }
    }
    const int64_t lo = (int64_t)layer * c->pool_rows;
    d->lv.k.data = c->kdata + lo * c->krow;
    d->lv.k.scales = c->ksb ? reinterpret_cast<uint16_t *>(c->kscales + lo * c->ksb) : nullptr;
    d->lv.v.data = c->vdata + lo * c->vrow;
    d->lv.v.scales = c->vsb ? reinterpret_cast<uint16_t *>(c->vscales + lo * c->vsb) : nullptr;
    d->pt = c->pt_dev + (int64_t)seq * c->max_pages;
    d->off = q.off;
    d->row0 = q.lfill[layer];
    d->P = c->P;
    return KVC_OK;
}

// Host bookkeeping of an append whose writes are enqueued.
static void append_commit(Ctx *c, int layer, int seq, int pos0, int n_tok, bool creates) {
    Seq &q = c->seqs[seq];
    if (creates) {
        q.linear = q.pos.empty() || (q.linear && (int64_t)q.pos.back() + 1 == pos0);
        for (int i = 0; i < n_tok; ++i) q.pos.push_back(pos0 + i);
        q.n += n_tok;
    }
    q.lfill[layer] += n_tok;
    c->recent[(size_t)seq][(size_t)layer] += n_tok;
}

static int append_impl(Ctx *c, int layer, int seq, int pos0, int n_tok, const float *k, const float *v,
                       void *stream, int in_heads) {
    if (n_tok < 1 || !k || !v) return c->fail(KVC_EINVAL, "n_tok must be >= 1 and k, v non-null");
    if (((uintptr_t)k | (uintptr_t)v) & 15) return c->fail(KVC_EINVAL, "k and v must be 16-byte aligned");
    bool creates = false;
    int rc = append_check(c, layer, seq, pos0, n_tok, &creates);
    if (rc) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    KVC_CU(c, cudaSetDevice(c->dev));
    if (c->host) {
        if (creates && (int64_t)c->seqs[seq].n + n_tok > c->P) return c->fail(KVC_ENOSPC, "host store is full");
        rc = transport_append(c, layer, n_tok, k, v, in_heads, st);
        if (rc) return rc;
    } else {
        AppendDst d;
        rc = device_append_dst(c, layer, seq, creates, n_tok, st, &d);
        if (rc) return rc;
        cudaError_t e = launch_append(c->tk, c->tv, c->Hk, in_heads, c->D, n_tok, k, v, &d, 1, st);
        if (e != cudaSuccess) return cuda_fail(c, e, "append kernel");
    }
    append_commit(c, layer, seq, pos0, n_tok, creates);
    return KVC_OK;
}

int kvc_attn_decode(kvc_ctx *cc, int layer, int n_seq, const int32_t *seq_ids, const float *q, float *out,
                    float kq_scale, void *stream) {
    if (!cc) return KVC_EINVAL;
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    if (c->split) {
        if (n_seq != 1 || !seq_ids || seq_ids[0] != 0)
            return c->fail(KVC_EINVAL, "split contexts attend sequence 0 only");
        if (!q || !out) return c->fail(KVC_EINVAL, "q and out must be non-null");
        // device heads first (they need no transfer), then the host heads, whose launch waits for
        // their delivery; query heads of a KV head are contiguous, so the two outputs sit side by side
        int rc = kvc_attn_decode(reinterpret_cast<kvc_ctx *>(c->part_dev), layer, 1, seq_ids, q, out, kq_scale,
                                 stream);
        if (rc) return c->fail(rc, c->part_dev->err);
        const int64_t skip = (int64_t)c->gpu_heads * c->r * c->D;
        rc = kvc_attn_decode(reinterpret_cast<kvc_ctx *>(c->part_host), layer, 1, seq_ids, q + skip, out + skip,
                             kq_scale, stream);
        if (rc) return c->fail(rc, c->part_host->err);
        return KVC_OK;
    }
    if (layer < 0 || layer >= c->L) return c->fail(KVC_EINVAL, "layer out of range");
    if (n_seq < 1 || !seq_ids || !q || !out) return c->fail(KVC_EINVAL, "n_seq >= 1 and non-null pointers required");
    if (!std::isfinite(kq_scale)) return c->fail(KVC_EINVAL, "kq_scale must be finite");
    if (q == out) return c->fail(KVC_EINVAL, "out may not alias q");
    if (((uintptr_t)q | (uintptr_t)out) & 15) return c->fail(KVC_EINVAL, "q and out must be 16-byte aligned");
    std::vector<char> seen(c->seqs.size(), 0);
    for (int i = 0; i < n_seq; ++i) {
        if (seq_ids[i] < 0 || seq_ids[i] >= (int)c->seqs.size()) return c->fail(KVC_EINVAL, "sequence id out of range");
        if (seen[(size_t)seq_ids[i]]) return c->fail(KVC_EINVAL, "duplicate sequence id");
        seen[(size_t)seq_ids[i]] = 1;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    KVC_CU(c, cudaSetDevice(c->dev));
    if (c->host) {
        if (n_seq != 1 || seq_ids[0] != 0) return c->fail(KVC_EINVAL, "host-resident contexts attend sequence 0 only");
        return transport_attn(c, layer, q, out, kq_scale, st);
    }
    std::vector<AttnSeq> seqs((size_t)n_seq);
    for (int i = 0; i < n_seq; ++i) {
        const Seq &s = c->seqs[(size_t)seq_ids[i]];
        AttnSeq &a = seqs[(size_t)i];
        a.page_table = c->pt_dev + (int64_t)seq_ids[i] * c->max_pages;
        a.off = s.off;
        a.n_rows = s.lfill[layer];
        a.out_row = i;
        a.stable_rows = std::max(0, a.n_rows - c->recent[(size_t)seq_ids[i]][(size_t)layer]);
        a.app_row = -1;
    }
    LayerView lv;
    const int64_t lo = (int64_t)layer * c->pool_rows;
    lv.k.data = c->kdata + lo * c->krow;
    lv.k.scales = c->ksb ? reinterpret_cast<uint16_t *>(c->kscales + lo * c->ksb) : nullptr;
    lv.v.data = c->vdata + lo * c->vrow;
    lv.v.scales = c->vsb ? reinterpret_cast<uint16_t *>(c->vscales + lo * c->vsb) : nullptr;
    const int64_t scale_limit = c->ksb ? c->kscale_bytes - lo * c->ksb : 0;
    int rc = launch_attention(c, lv, &c->tmk[2 * (size_t)layer], &c->tmv[2 * (size_t)layer], c->P, scale_limit, n_seq,
                              seqs.data(), q, out, kq_scale, st);
    if (rc == KVC_OK) c->clear_recent(); // kernels after this one start only once it has waited
    return rc;
}

int kvc_decode_step(kvc_ctx *cc, int layer, int n_seq, const int32_t *seq_ids, const int32_t *pos, const float *k,
                    const float *v, const float *q, float *out, float kq_scale, void *stream) {
    if (!cc) return KVC_EINVAL;
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    if (n_seq < 1 || !seq_ids || !pos || !k || !v || !q || !out)
        return c->fail(KVC_EINVAL, "n_seq >= 1 and non-null pointers required");
    if (((uintptr_t)k | (uintptr_t)v) & 15) return c->fail(KVC_EINVAL, "k and v must be 16-byte aligned");
    if (c->split || c->host) {
        // one sequence; the append and the attention as two launches (the rows go through the
        // host store and the staging ring)
        if (n_seq != 1 || seq_ids[0] != 0) return c->fail(KVC_EINVAL, "this context decodes sequence 0 only");
        int rc = kvc_append(cc, layer, 0, pos[0], 1, k, v, stream);
        if (rc) return rc;
        return kvc_attn_decode(cc, layer, 1, seq_ids, q, out, kq_scale, stream);
    }
    if (layer < 0 || layer >= c->L) return c->fail(KVC_EINVAL, "layer out of range");
    if (!std::isfinite(kq_scale)) return c->fail(KVC_EINVAL, "kq_scale must be finite");
    if (q == out) return c->fail(KVC_EINVAL, "out may not alias q");
    if (((uintptr_t)q | (uintptr_t)out) & 15) return c->fail(KVC_EINVAL, "q and out must be 16-byte aligned");
    std::vector<char> seen(c->seqs.size(), 0);
    std::vector<char> creates((size_t)n_seq, 0);
    int64_t new_pages = 0;
    for (int i = 0; i < n_seq; ++i) {
        const int id = seq_ids[i];
        if (id < 0 || id >= (int)c->seqs.size()) return c->fail(KVC_EINVAL, "sequence id out of range");
        if (seen[(size_t)id]) return c->fail(KVC_EINVAL, "duplicate sequence id");
        seen[(size_t)id] = 1;
        bool cr = false;
        int rc = append_check(c, layer, id, pos[i], 1, &cr);
        if (rc) return rc;
        creates[(size_t)i] = cr;
        if (cr) {
            const Seq &s = c->seqs[(size_t)id];
            const int32_t need = pages_for(c, s.off, (int64_t)s.n + 1);
            if (need > c->max_pages) return c->fail(KVC_ENOSPC, "sequence would exceed the page table");
            new_pages += std::max<int64_t>(0, need - (int64_t)s.pages.size());
        }
    }
    if (new_pages > (int64_t)c->free_pages.size()) return c->fail(KVC_ENOSPC, "no free pages");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    KVC_CU(c, cudaSetDevice(c->dev));
    // cells and page-table entries first (the checks above leave nothing to fail but CUDA)
    for (int i = 0; i < n_seq; ++i) {
        AppendDst d;
        int rc = device_append_dst(c, layer, seq_ids[i], creates[(size_t)i] != 0, 1, st, &d);
        if (rc) return rc;
        append_commit(c, layer, seq_ids[i], pos[i], 1, creates[(size_t)i] != 0);
    }
    std::vector<AttnSeq> seqs((size_t)n_seq);
    for (int i = 0; i < n_seq; ++i) {
        const Seq &s = c->seqs[(size_t)seq_ids[i]];
        AttnSeq &a = seqs[(size_t)i];
        a.page_table = c->pt_dev + (int64_t)seq_ids[i] * c->max_pages;
        a.off = s.off;
        a.n_rows = s.lfill[layer];
        a.out_row = i;
        a.stable_rows = std::max(0, a.n_rows - c->recent[(size_t)seq_ids[i]][(size_t)layer]);
        a.app_row = a.n_rows - 1;
    }
    LayerView lv;
    const int64_t lo = (int64_t)layer * c->pool_rows;
    lv.k.data = c->kdata + lo * c->krow;
    lv.k.scales = c->ksb ? reinterpret_cast<uint16_t *>(c->kscales + lo * c->ksb) : nullptr;
    lv.v.data = c->vdata + lo * c->vrow;
    lv.v.scales = c->vsb ? reinterpret_cast<uint16_t *>(c->vscales + lo * c->vsb) : nullptr;
    const int64_t scale_limit = c->ksb ? c->kscale_bytes - lo * c->ksb : 0;
    int rc = launch_attention(c, lv, &c->tmk[2 * (size_t)layer], &c->tmv[2 * (size_t)layer], c->P, scale_limit, n_seq,
                              seqs.data(), q, out, kq_scale, st, k, v);
    if (rc) return rc;
    // Everything before this launch is complete once the next kernel starts, but the new rows
    // are stored after this kernel lets the next one start: they stay recent for it.
    c->clear_recent();
    for (int i = 0; i < n_seq; ++i) c->recent[(size_t)seq_ids[i]][(size_t)layer] = 1;
    return KVC_OK;
}

int kvc_seq_rm(kvc_ctx *cc, int seq, int p0, int p1) {
    if (!cc) return KVC_EINVAL;
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    if (c->host) return c->fail(KVC_EINVAL, "sequence operations need a device-resident context");
    if (seq < 0 || seq >= (int)c->seqs.size()) return c->fail(KVC_EINVAL, "sequence id out of range");
    Seq &q = c->seqs[(size_t)seq];
    if (!q.synced()) return c->fail(KVC_EINVAL, "layers are not in sync (a step's appends are incomplete)");
    int64_t a, b;
    norm_range(p0, p1, a, b);
    RowSel rm;
    select_rows(q, a, b, rm);
    if (rm.count == 0) return KVC_OK;
    int rc = enter_sync(c);
    if (rc) return rc;
    const int64_t k = rm.count;
    const bool prefix = rm.contiguous && rm.first == 0;
    const bool suffix = rm.contiguous && rm.first + k == q.n;
    if (k == q.n) {
        q.n = 0;
        q.pos.clear();
        q.linear = true;
        release_tail_pages(c, q);
    } else if (prefix) {
        q.off += (int32_t)k;
        q.n -= (int32_t)k;
        q.pos.erase(q.pos.begin(), q.pos.begin() + k);
        int32_t drop = q.off / c->P;
        for (int32_t i = 0; i < drop; ++i) c->free_pages.push_back(q.pages[(size_t)i]);
        q.pages.erase(q.pages.begin(), q.pages.begin() + drop);
        q.off -= drop * c->P;
        q.dev_pages = 0;
    } else if (suffix) {
        q.n -= (int32_t)k;
        q.pos.resize((size_t)q.n);
        release_tail_pages(c, q);
    } else {
        // compact: kept rows from the first removed row on go through staging
        const int64_t i0 = rm.first;
        RowSel keep;
        if (rm.contiguous) {
            keep = row_range(i0 + k, q.n - i0 - k);
        } else {
            keep.contiguous = false;
            size_t j = 0;
            for (int64_t r = i0; r < q.n; ++r) {
                if (j < rm.idx.size() && rm.idx[j] == r) {
                    ++j;
                    continue;
                }
                keep.idx.push_back(r);
            }
            keep.count = (int64_t)keep.idx.size();
        }
        const int64_t nk = keep.count;
        if ((rc = ensure_staging(c, payload_bytes(c, nk)))) return rc;
        // pack the kept rows, then unpack them at logical rows i0 .. i0+nk-1
        std::vector<RowRun> runs;
        add_payload_copies(c, q, keep, runs);
        if ((rc = upload_runs(c, runs))) return rc;
        KVC_CU(c, launch_copy_runs(payload_args(c, nk, c->staging, true), c->runs_dev, (int64_t)runs.size(), c->L,
                                   c->st));
        if ((rc = wait_internal(c))) return rc;
        runs.clear();
        add_payload_copies(c, q, row_range(i0, nk), runs);
        if ((rc = upload_runs(c, runs))) return rc;
        KVC_CU(c, launch_copy_runs(payload_args(c, nk, c->staging, false), c->runs_dev, (int64_t)runs.size(), c->L,
                                   c->st));
        if ((rc = wait_internal(c))) return rc;
        std::vector<int32_t> np;
        np.reserve((size_t)(q.n - k));
        np.insert(np.end(), q.pos.begin(), q.pos.begin() + i0);
        for (int64_t i = 0; i < nk; ++i) np.push_back(q.pos[(size_t)keep.row(i)]);
        q.pos.swap(np);
        q.n -= (int32_t)k;
        q.linear = consecutive(q.pos.data(), q.n);
        release_tail_pages(c, q);
    }
    for (auto &f : q.lfill) f = q.n;
    if ((rc = upload_pages(c, seq))) return rc;
    return wait_internal(c);
}

int kvc_seq_cp(kvc_ctx *cc, int src, int dst, int p0, int p1) {
    if (!cc) return KVC_EINVAL;
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    if (c->host) return c->fail(KVC_EINVAL, "sequence operations need a device-resident context");
    if (src < 0 || src >= (int)c->seqs.size() || dst < 0 || dst >= (int)c->seqs.size())
        return c->fail(KVC_EINVAL, "sequence id out of range");
    if (src == dst) return KVC_OK;
    Seq &a = c->seqs[(size_t)src];
    Seq &b = c->seqs[(size_t)dst];
    if (!a.synced() || !b.synced()) return c->fail(KVC_EINVAL, "layers are not in sync");
    int64_t lo, hi;
    norm_range(p0, p1, lo, hi);
    RowSel sel;
    select_rows(a, lo, hi, sel);
    if (sel.count == 0) return KVC_OK;
    int rc = enter_sync(c);
    if (rc) return rc;
    size_t first_new;
    if ((rc = grow_pages(c, b, sel.count, &first_new))) return rc;
    const int64_t base = b.n;
    b.n += (int32_t)sel.count;
    std::vector<RowRun> runs;
    if (sel.contiguous) {
        b.pos.insert(b.pos.end(), a.pos.begin() + sel.first, a.pos.begin() + sel.first + sel.count);
        add_row_copies(c, a, sel.first, b, base, sel.count, runs);
    } else {
        for (int64_t r : sel.idx) b.pos.push_back(a.pos[(size_t)r]);
        for (size_t i = 0; i < sel.idx.size();) {
            size_t j = i + 1;
            while (j < sel.idx.size() && sel.idx[j] == sel.idx[j - 1] + 1) ++j;
            add_row_copies(c, a, sel.idx[i], b, base + (int64_t)i, (int64_t)(j - i), runs);
            i = j;
        }
    }
    const bool copied_linear = (a.linear && sel.contiguous) || consecutive(b.pos.data() + base, sel.count);
    b.linear = (base == 0 || (b.linear && (int64_t)b.pos[(size_t)base - 1] + 1 == b.pos[(size_t)base])) &&
               copied_linear;
    for (auto &f : b.lfill) f = b.n;
    if ((rc = upload_pages(c, dst))) return rc;
    if ((rc = upload_runs(c, runs))) return rc;
    KVC_CU(c, launch_copy_runs(pool_args(c), c->runs_dev, (int64_t)runs.size(), c->L, c->st));
    return wait_internal(c);
}

int kvc_seq_add(kvc_ctx *cc, int seq, int p0, int p1, int delta) {
    if (!cc) return KVC_EINVAL;
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    if (c->host) return c->fail(KVC_EINVAL, "sequence operations need a device-resident context");
    if (seq < 0 || seq >= (int)c->seqs.size()) return c->fail(KVC_EINVAL, "sequence id out of range");
    Seq &q = c->seqs[(size_t)seq];
    if (!q.synced()) return c->fail(KVC_EINVAL, "layers are not in sync");
    int64_t a, b;
    norm_range(p0, p1, a, b);
    if (delta == 0) return KVC_OK;
    RowSel sel;
    select_rows(q, a, b, sel);
    if (sel.count == 0) return KVC_OK;
    if (sel.pos_min + delta < 0 || sel.pos_max + delta > INT32_MAX)
        return c->fail(KVC_ERANGE, "shifted position out of range");
    // runs of consecutive cells inside one page, one span per KV head (layer
    // 0; the kernel repeats them for every layer), at most ROPE_SPAN_MAX rows
    std::vector<RopeSpan> &spans = c->spans_host;
    spans.clear();
    for (int64_t i = 0; i < sel.count;) {
        int32_t pg, cl;
        phys(c, q, sel.row(i), pg, cl);
        int64_t j = std::min<int64_t>({sel.count, i + ROPE_SPAN_MAX, i + (c->P - cl)});
        if (!sel.contiguous)
            for (int64_t m = i + 1; m < j; ++m)
                if (sel.idx[(size_t)m] != sel.idx[(size_t)m - 1] + 1) {
                    j = m;
                    break;
                }
        for (int g = 0; g < c->Hk; ++g) spans.push_back(RopeSpan{prow(c, pg, g, cl), (int32_t)(j - i), 0});
        i = j;
    }
    int rc = enter_sync(c);
    if (rc) return rc;
    const int64_t n_spans = (int64_t)spans.size();
    if (n_spans > c->spans_cap) {
        dev_free(c, c->spans_dev, c->spans_cap * (int64_t)sizeof(RopeSpan));
        c->spans_dev = nullptr;
        c->spans_cap = 0;
        if ((rc = dev_alloc(c, (void **)&c->spans_dev, n_spans * (int64_t)sizeof(RopeSpan), "span list")))
            return rc;
        c->spans_cap = n_spans;
    }
    if ((rc = upload(c, c->spans_dev, spans.data(), (int64_t)(spans.size() * sizeof(RopeSpan))))) return rc;
    // cos/sin of delta * theta_i in fp64, theta_i = base^(-2i/D)
    float2 cs[64];
    for (int i = 0; i < c->D / 2; ++i) {
        const double theta = std::pow((double)c->prm.rope_base, -2.0 * i / (double)c->D);
        const double phi = (double)delta * theta;
        cs[i] = make_float2((float)std::cos(phi), (float)std::sin(phi));
    }
    cudaError_t e = launch_rope_shift(c->tk, c->D, c->prm.rope_mode, c->kdata,
                                      reinterpret_cast<uint16_t *>(c->kscales), c->pool_rows, c->L, c->spans_dev,
                                      n_spans, cs, c->err_dev, c->st);
    if (e != cudaSuccess) return cuda_fail(c, e, "rope shift kernel");
    if ((rc = wait_internal(c))) return rc;
    int32_t *pos = q.pos.data();
    if (sel.contiguous)
        for (int64_t r = sel.first; r < sel.first + sel.count; ++r) pos[r] += delta;
    else
        for (int64_t r : sel.idx) pos[r] += delta;
    if (!(sel.contiguous && sel.first == 0 && sel.count == q.n)) q.linear = consecutive(pos, q.n);
    return KVC_OK;
}

int kvc_seq_key_scores(kvc_ctx *cc, int seq, int layer, float *scores, int32_t cap, int32_t *n) {
    if (!cc || !n) return KVC_EINVAL;
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    if (c->host) return c->fail(KVC_EINVAL, "sequence operations need a device-resident context");
    if (seq < 0 || seq >= (int)c->seqs.size()) return c->fail(KVC_EINVAL, "sequence id out of range");
    if (layer < 0) layer = c->L / 2;
    if (layer >= c->L) return c->fail(KVC_EINVAL, "layer out of range");
    Seq &q = c->seqs[(size_t)seq];
    if (!q.synced()) return c->fail(KVC_EINVAL, "layers are not in sync");
    const int64_t rows = q.n;
    *n = (int32_t)rows;
    if (!scores) return KVC_OK;
    if (cap < rows) return c->fail(KVC_ENOSPC, "score buffer too small");
    if (rows == 0) return KVC_OK;
    int rc = enter_sync(c);
    if (rc) return rc;
    // the rows in storage order as blocks of consecutive rows of one page;
    // the scores come back in that order and are put in position order here
    std::vector<KeyDiffBlock> blocks;
    const int br = keydiff_block_rows(c->tk == KVC_Q8_0, c->Hk, c->D);
    for (int64_t i = 0; i < rows;) {
        int32_t pg, cl;
        phys(c, q, i, pg, cl);
        const int64_t n = std::min<int64_t>({(int64_t)br, rows - i, (int64_t)(c->P - cl)});
        blocks.push_back(KeyDiffBlock{prow(c, pg, 0, cl), (int32_t)n, (int32_t)i});
        i += n;
    }
    const int64_t nb = (int64_t)blocks.size();
    const int64_t slices = (nb + keydiff_slice_blocks() - 1) / keydiff_slice_blocks();
    auto al = [](int64_t x) { return (x + 255) / 256 * 256; };
    const int64_t o_blocks = 0, o_sum = al(nb * (int64_t)sizeof(KeyDiffBlock));
    const int64_t o_mean = o_sum + al((int64_t)c->Hk * slices * c->D * 4);
    const int64_t o_norm = o_mean + al((int64_t)c->Hk * c->D * 4), o_score = o_norm + al((int64_t)c->Hk * 4);
    if ((rc = ensure_staging(c, o_score + al(rows * 4)))) return rc;
    uint8_t *w = c->staging;
    if ((rc = upload(c, w + o_blocks, blocks.data(), (int64_t)(blocks.size() * sizeof(KeyDiffBlock))))) return rc;
    KeyDiffArgs a;
    std::memset(&a, 0, sizeof(a));
    a.q8 = c->tk == KVC_Q8_0;
    a.Hk = c->Hk;
    a.D = c->D;
    a.P = c->P;
    a.kdata = c->kdata;
    a.kscales = a.q8 ? reinterpret_cast<const uint16_t *>(c->kscales) : nullptr;
    a.layer_off = (int64_t)layer * c->pool_rows;
    a.blocks = reinterpret_cast<const KeyDiffBlock *>(w + o_blocks);
    a.n_blocks = (int32_t)nb;
    a.block_rows = br;
    a.n_slices = (int32_t)slices;
    a.n_rows = rows;
    a.slice_sum = reinterpret_cast<float *>(w + o_sum);
    a.mean = reinterpret_cast<float *>(w + o_mean);
    a.mean_norm = reinterpret_cast<float *>(w + o_norm);
    a.score = reinterpret_cast<float *>(w + o_score);
    a.err = c->err_dev;
    cudaError_t e = launch_keydiff(a, c->sms, c->st);
    if (e != cudaSuccess) return cuda_fail(c, e, "KeyDiff kernels");
    if (q.linear || std::is_sorted(q.pos.begin(), q.pos.end())) {
        KVC_CU(c, cudaMemcpyAsync(scores, w + o_score, (size_t)rows * 4, cudaMemcpyDeviceToHost, c->st));
        return wait_internal(c);
    }
    std::vector<float> tmp((size_t)rows);
    KVC_CU(c, cudaMemcpyAsync(tmp.data(), w + o_score, (size_t)rows * 4, cudaMemcpyDeviceToHost, c->st));
    if ((rc = wait_internal(c))) return rc;
    std::vector<int64_t> order((size_t)rows);
    for (int64_t r = 0; r < rows; ++r) order[(size_t)r] = r;
    std::stable_sort(order.begin(), order.end(),
                     [&](int64_t x, int64_t y) { return q.pos[(size_t)x] < q.pos[(size_t)y]; });
    for (int64_t j = 0; j < rows; ++j) scores[j] = tmp[(size_t)order[(size_t)j]];
    return KVC_OK;
}

int kvc_seq_evict_window(kvc_ctx *cc, int seq, int layer, int n_keep, int n_discard, int n_recent, int32_t *p0) {
    if (!cc || !p0) return KVC_EINVAL;
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    if (n_discard < 1 || n_keep < 0 || n_recent < 0) return c->fail(KVC_EINVAL, "bad window arguments");
    *p0 = -1;
    int32_t n = 0;
    int rc = kvc_seq_key_scores(cc, seq, layer, nullptr, 0, &n);
    if (rc) return rc;
    std::vector<float> sc((size_t)n);
    if (n > 0 && (rc = kvc_seq_key_scores(cc, seq, layer, sc.data(), n, &n))) return rc;
    // smallest window sum by prefix sums in fp64 (the first on ties)
    const int64_t lo = n_keep, hi = (int64_t)n - n_recent, wd = n_discard;
    if (hi - lo < wd) return KVC_OK;
    std::vector<double> pre((size_t)n + 1, 0.0);
    for (int64_t j = 0; j < n; ++j) pre[(size_t)j + 1] = pre[(size_t)j] + (double)sc[(size_t)j];
    int64_t best = lo;
    double best_sum = pre[(size_t)(lo + wd)] - pre[(size_t)lo];
    for (int64_t s = lo + 1; s + wd <= hi; ++s) {
        const double sum = pre[(size_t)(s + wd)] - pre[(size_t)s];
        if (sum < best_sum) {
            best_sum = sum;
            best = s;
        }
    }
    Seq &q = c->seqs[(size_t)seq];
    std::vector<int32_t> pos(q.pos.begin(), q.pos.end());
    std::stable_sort(pos.begin(), pos.end());
    const int32_t first = pos[(size_t)best], last = pos[(size_t)(best + wd - 1)];
    if ((rc = kvc_seq_rm(cc, seq, first, last + 1))) return rc;
    if ((rc = kvc_seq_add(cc, seq, last + 1, -1, -(last + 1 - first)))) return rc;
    *p0 = first;
    return KVC_OK;
}

int kvc_state_get(kvc_ctx *cc, int seq, int p0, int p1, void *dst, size_t cap, size_t *n_written) {
    if (!cc) return KVC_EINVAL;
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    if (c->host) return c->fail(KVC_EINVAL, "state operations need a device-resident context");
    if (seq < 0 || seq >= (int)c->seqs.size() || !n_written) return c->fail(KVC_EINVAL, "bad sequence id or n_written");
    Seq &q = c->seqs[(size_t)seq];
    if (!q.synced()) return c->fail(KVC_EINVAL, "layers are not in sync");
    int64_t a, b;
    norm_range(p0, p1, a, b);
    RowSel sel;
    select_rows(q, a, b, sel);
    const int64_t n = sel.count;
    const int64_t size = state_bytes(c, n);
    *n_written = (size_t)size;
    if (!dst) return KVC_OK;
    if ((int64_t)cap < size) return c->fail(KVC_ENOSPC, "destination buffer too small");
    int rc = enter_sync(c);
    if (rc) return rc;
    uint8_t *out = reinterpret_cast<uint8_t *>(dst);
    std::memset(out, 0, (size_t)(64 + pad16(4 * n)));
    uint32_t hdr[8] = {0x3143564Bu, 1u, (uint32_t)c->L, (uint32_t)c->Hk, (uint32_t)c->D,
                       (uint32_t)c->tk, (uint32_t)c->tv, (uint32_t)n};
    std::memcpy(out, hdr, sizeof(hdr));
    const uint64_t pl = (uint64_t)payload_bytes(c, n);
    std::memcpy(out + 32, &pl, 8);
    if (sel.contiguous)
        std::memcpy(out + 64, q.pos.data() + sel.first, (size_t)(4 * n));
    else
        for (int64_t i = 0; i < n; ++i) std::memcpy(out + 64 + 4 * i, &q.pos[(size_t)sel.idx[(size_t)i]], 4);
    if (n > 0) {
        if ((rc = ensure_staging(c, (int64_t)pl))) return rc;
        if ((rc = ensure_copy_stream(c))) return rc;
        std::vector<RowRun> runs;
        add_payload_copies(c, q, sel, runs);
        if ((rc = upload_runs(c, runs))) return rc;
        const RunCopyArgs ca = payload_args(c, n, c->staging, true);
        // pack a layer group on st, then copy it to the host on st_copy while
        // the next group is packed
        uint8_t *hp = out + 64 + pad16(4 * n);
        const int64_t per_layer = section_bytes(c, c->tk, n) + section_bytes(c, c->tv, n);
        const int k = state_chunks(c);
        for (int i = 0; i < k; ++i) {
            const int l0 = chunk_layer(c, i), l1 = chunk_layer(c, i + 1);
            RunCopyArgs cl = ca;
            cl.l0 = l0;
            KVC_CU(c, launch_copy_runs(cl, c->runs_dev, (int64_t)runs.size(), l1 - l0, c->st));
            KVC_CU(c, cudaEventRecord(c->st_ev[i], c->st));
            KVC_CU(c, cudaStreamWaitEvent(c->st_copy, c->st_ev[i], 0));
            KVC_CU(c, cudaMemcpyAsync(hp + l0 * per_layer, c->staging + l0 * per_layer, (size_t)((l1 - l0) * per_layer),
                                      cudaMemcpyDeviceToHost, c->st_copy));
        }
        KVC_CU(c, cudaEventRecord(c->st_ev[Ctx::STATE_CHUNKS], c->st_copy));
        KVC_CU(c, cudaStreamWaitEvent(c->st, c->st_ev[Ctx::STATE_CHUNKS], 0));
        if ((rc = wait_internal(c))) return rc;
        zero_payload_pads(c, hp, n); // the staging buffer's padding bytes are not written
    }
    return KVC_OK;
}

int kvc_state_set(kvc_ctx *cc, int seq, const void *src, size_t nbytes, size_t *n_read) {
    if (!cc) return KVC_EINVAL;
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    if (c->host) return c->fail(KVC_EINVAL, "state operations need a device-resident context");
    if (seq < 0 || seq >= (int)c->seqs.size() || !src) return c->fail(KVC_EINVAL, "bad sequence id or source");
    Seq &q = c->seqs[(size_t)seq];
    if (!q.synced()) return c->fail(KVC_EINVAL, "layers are not in sync");
    const uint8_t *in = reinterpret_cast<const uint8_t *>(src);
    if (nbytes < 64) return c->fail(KVC_EFORMAT, "state shorter than its header");
    uint32_t hdr[8];
    uint64_t pl;
    std::memcpy(hdr, in, sizeof(hdr));
    std::memcpy(&pl, in + 32, 8);
    if (hdr[0] != 0x3143564Bu || hdr[1] != 1u) return c->fail(KVC_EFORMAT, "bad magic or version");
    if (hdr[2] != (uint32_t)c->L || hdr[3] != (uint32_t)c->Hk || hdr[4] != (uint32_t)c->D ||
        hdr[5] != (uint32_t)c->tk || hdr[6] != (uint32_t)c->tv)
        return c->fail(KVC_EFORMAT, "state geometry or types differ from this context");
    const int64_t n = (int64_t)hdr[7];
    if (n > INT32_MAX) return c->fail(KVC_EFORMAT, "bad token count");
    if (pl != (uint64_t)payload_bytes(c, n)) return c->fail(KVC_EFORMAT, "payload size does not match the header");
    const int64_t size = state_bytes(c, n);
    if ((int64_t)nbytes < size) return c->fail(KVC_EFORMAT, "state truncated");
    std::vector<int32_t> pos((size_t)n);
    for (int64_t i = 0; i < n; ++i) {
        std::memcpy(&pos[(size_t)i], in + 64 + 4 * i, 4);
        if (pos[(size_t)i] < 0) return c->fail(KVC_EFORMAT, "negative position in state");
    }
    if (n_read) *n_read = (size_t)size;
    if (n == 0) return KVC_OK;
    int rc = enter_sync(c);
    if (rc) return rc;
    size_t first_new;
    if ((rc = grow_pages(c, q, n, &first_new))) return rc;
    if ((rc = ensure_staging(c, (int64_t)pl))) {
        release_tail_pages(c, q);
        return rc;
    }
    const int64_t base = q.n;
    q.n += (int32_t)n;
    q.pos.insert(q.pos.end(), pos.begin(), pos.end());
    q.linear = (base == 0 || (q.linear && (int64_t)q.pos[(size_t)base - 1] + 1 == q.pos[(size_t)base])) &&
               consecutive(pos.data(), n);
    for (auto &f : q.lfill) f = q.n;
    std::vector<RowRun> runs;
    add_payload_copies(c, q, row_range(base, n), runs);
    if ((rc = upload_pages(c, seq))) return rc;
    if ((rc = upload_runs(c, runs))) return rc;
    const RunCopyArgs ca = payload_args(c, n, c->staging, false);
    if ((rc = ensure_copy_stream(c))) return rc;
    // copy a layer group to the device on st_copy, unpack it on st while the
    // next group is copied (the staging buffer is idle: enter_sync waited)
    const uint8_t *hp = in + 64 + pad16(4 * n);
    const int64_t per_layer = section_bytes(c, c->tk, n) + section_bytes(c, c->tv, n);
    const int k = state_chunks(c);
    for (int i = 0; i < k; ++i) {
        const int l0 = chunk_layer(c, i), l1 = chunk_layer(c, i + 1);
        RunCopyArgs cl = ca;
        cl.l0 = l0;
        KVC_CU(c, cudaMemcpyAsync(c->staging + l0 * per_layer, hp + l0 * per_layer, (size_t)((l1 - l0) * per_layer),
                                  cudaMemcpyHostToDevice, c->st_copy));
        KVC_CU(c, cudaEventRecord(c->st_ev[i], c->st_copy));
        KVC_CU(c, cudaStreamWaitEvent(c->st, c->st_ev[i], 0));
        KVC_CU(c, launch_copy_runs(cl, c->runs_dev, (int64_t)runs.size(), l1 - l0, c->st));
    }
    return wait_internal(c);
}

int kvc_pipeline_depth(kvc_ctx *cc, int n) {
    if (!cc) return KVC_EINVAL;
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    if (c->split) {
        int rc = kvc_pipeline_depth(reinterpret_cast<kvc_ctx *>(c->part_host), n);
        return rc ? c->fail(rc, c->part_host->err) : KVC_OK;
    }
    if (n < 0 || n > 16) return c->fail(KVC_EINVAL, "depth must be in [0, 16]");
    if (c->host) {
        cudaSetDevice(c->dev);
        cudaDeviceSynchronize();
        transport_release(c);
        c->tr.latched = false;
    }
    c->tr.depth = n;
    return KVC_OK;
}

int kvc_pipeline_budget(kvc_ctx *cc, size_t bytes) {
    if (!cc) return KVC_EINVAL;
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    if (c->split) {
        int rc = kvc_pipeline_budget(reinterpret_cast<kvc_ctx *>(c->part_host), bytes);
        return rc ? c->fail(rc, c->part_host->err) : KVC_OK;
    }
    if (bytes > ((size_t)1 << 50)) return c->fail(KVC_EINVAL, "budget too large");
    if (c->host) {
        cudaSetDevice(c->dev);
        cudaDeviceSynchronize();
        transport_release(c);
        c->tr.latched = false;
    }
    c->tr.budget = (int64_t)bytes;
    return KVC_OK;
}

int kvc_seq_n_tokens(const kvc_ctx *cc, int seq, int32_t *n) {
    if (!cc || !n) return KVC_EINVAL;
    const Ctx *c = reinterpret_cast<const Ctx *>(cc);
    if (c->split) return kvc_seq_n_tokens(reinterpret_cast<const kvc_ctx *>(c->part_dev), seq, n);
    if (seq < 0 || seq >= (int)c->seqs.size()) return KVC_EINVAL;
    *n = c->seqs[(size_t)seq].n;
    return KVC_OK;
}

int kvc_seq_positions(const kvc_ctx *cc, int seq, int32_t *pos, int32_t cap, int32_t *n) {
    if (!cc || !n) return KVC_EINVAL;
    const Ctx *c = reinterpret_cast<const Ctx *>(cc);
    if (c->split) return kvc_seq_positions(reinterpret_cast<const kvc_ctx *>(c->part_dev), seq, pos, cap, n);
    if (seq < 0 || seq >= (int)c->seqs.size()) return KVC_EINVAL;
    const Seq &q = c->seqs[(size_t)seq];
    *n = q.n;
    if (pos) {
        if (cap < q.n) return KVC_ENOSPC;
        std::memcpy(pos, q.pos.data(), (size_t)q.n * 4);
    }
    return KVC_OK;
}

int kvc_get_stats(const kvc_ctx *cc, kvc_stats *o) {
    if (!cc || !o) return KVC_EINVAL;
    const Ctx *c = reinterpret_cast<const Ctx *>(cc);
    if (c->split) {
        // the transport is the host half's; memory is both halves'
        kvc_get_stats(reinterpret_cast<const kvc_ctx *>(c->part_host), o);
        kvc_stats d;
        kvc_get_stats(reinterpret_cast<const kvc_ctx *>(c->part_dev), &d);
        o->pages_total = d.pages_total;
        o->pages_free = d.pages_free;
        o->device_bytes += d.device_bytes;
        return KVC_OK;
    }
    std::memset(o, 0, sizeof(*o));
    o->ring_engaged = c->tr.ring.empty() ? 0 : 1;
    o->ring_declined = c->tr.latched ? 1 : 0;
    o->ring_slots = (int32_t)c->tr.ring.size();
    o->transfer_stream = c->tr.xfer ? 1 : 0;
    o->slot_bytes = c->tr.ring.empty() ? c->tr.ordered.bytes : c->tr.ring[0].bytes;
    for (auto &s : c->tr.ring) o->ring_bytes += s.bytes;
    o->ordered_bytes = c->tr.ordered.bytes;
    o->deliveries_early = c->tr.early;
    o->deliveries_ordered = c->tr.in_order;
    o->bytes_delivered = c->tr.bytes;
    o->pages_total = c->n_pages;
    o->pages_free = (int64_t)c->free_pages.size();
    o->device_bytes = c->device_bytes;
    o->host_pinned_bytes = c->host_bytes;
    o->rolling = c->tr.rolling ? 1 : 0;
    o->tile_rows = c->tr.rolling && !c->tr.ring.empty() ? c->tr.ring[0].cap : 0;
    o->tiles_delivered = c->tr.tiles;
    return KVC_OK;
}

int kvc_set_chunk_rows(kvc_ctx *cc, int rows) {
    if (!cc) return KVC_EINVAL;
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    if (c->split) {
        int rc = kvc_set_chunk_rows(reinterpret_cast<kvc_ctx *>(c->part_dev), rows);
        if (!rc) rc = kvc_set_chunk_rows(reinterpret_cast<kvc_ctx *>(c->part_host), rows);
        return rc ? c->fail(rc, "bad chunk rows") : KVC_OK;
    }
    if (rows < 0 || rows % 16) return c->fail(KVC_EINVAL, "chunk rows must be a non-negative multiple of 16");
    c->chunk_override = rows;
    return KVC_OK;
}

int kvc_set_timeout_ms(kvc_ctx *cc, int ms) {
    if (!cc) return KVC_EINVAL;
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    if (c->split) {
        int rc = kvc_set_timeout_ms(reinterpret_cast<kvc_ctx *>(c->part_dev), ms);
        if (!rc) rc = kvc_set_timeout_ms(reinterpret_cast<kvc_ctx *>(c->part_host), ms);
        return rc ? c->fail(rc, "bad timeout") : KVC_OK;
    }
    if (ms < 1) return c->fail(KVC_EINVAL, "timeout must be positive");
    c->timeout_ms = ms;
    return KVC_OK;
}

int kvc_debug_select_rows(const int32_t *pos, int32_t n, int linear, int p0, int p1, int64_t *rows,
                          int64_t *count, int64_t *first, int32_t *contiguous) {
    if (n < 0 || (n > 0 && !pos) || !count || !first || !contiguous) return KVC_EINVAL;
    Seq q;
    q.n = n;
    q.pos.assign(pos, pos + n);
    for (int32_t r = 0; r < n; ++r)
        if (q.pos[(size_t)r] < 0) return KVC_EINVAL;
    q.linear = linear != 0;
    if (q.linear && !consecutive(q.pos.data(), n)) return KVC_EINVAL;
    int64_t a, b;
    norm_range(p0, p1, a, b);
    RowSel sel;
    select_rows(q, a, b, sel);
    *count = sel.count;
    *first = sel.count ? sel.first : 0;
    *contiguous = sel.contiguous ? 1 : 0;
    if (rows)
        for (int64_t i = 0; i < sel.count; ++i) rows[i] = sel.row(i);
    return KVC_OK;
}

int kvc_debug_fail_alloc_after(kvc_ctx *cc, int n) {
    if (!cc) return KVC_EINVAL;
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    if (c->split) {
        kvc_debug_fail_alloc_after(reinterpret_cast<kvc_ctx *>(c->part_dev), n);
        kvc_debug_fail_alloc_after(reinterpret_cast<kvc_ctx *>(c->part_host), n);
        return KVC_OK;
    }
    c->fail_after = n < 0 ? -1 : n;
    return KVC_OK;
}

int kvc_check_device_error(kvc_ctx *cc, uint32_t *word) {
    if (!cc || !word) return KVC_EINVAL;
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    if (c->split) {
        uint32_t a = 0, b = 0;
        int rc = kvc_check_device_error(reinterpret_cast<kvc_ctx *>(c->part_dev), &a);
        if (!rc) rc = kvc_check_device_error(reinterpret_cast<kvc_ctx *>(c->part_host), &b);
        *word = a | b;
        return rc;
    }
    KVC_CU(c, cudaSetDevice(c->dev));
    KVC_CU(c, cudaDeviceSynchronize());
    KVC_CU(c, cudaMemcpy(word, c->err_dev, 4, cudaMemcpyDeviceToHost));
    KVC_CU(c, cudaMemsetAsync(c->err_dev, 0, 4, c->st)); // the internal stream is non-blocking: wait for it
    KVC_CU(c, cudaStreamSynchronize(c->st));
    return KVC_OK;
}

} // extern "C"
