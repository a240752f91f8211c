// transport.cu - split-K launch planning and the host-resident transport.
//
// Host-resident KV ("sched: pipeline the delivery of a host-resident KV
// cache (R4)", section What it does) keeps each layer's K/V in pinned host
// memory.  Before a layer's attention its rows reach the device through a
// staging ring of N+2 slots that lives outside any allocator, each slot
// holding one layer's K+V over the context, with a ready/release event pair:
//  1. stable prefix: a delivery carries the rows the layer holds when it is
//     issued; rows written later in the step (the token being appended) are
//     written into the slot by the append itself, so no delivery ever has to
//     wait for them (item 1);
//  2. the ring: delivery of layer l+N is issued right after the attention of
//     layer l is enqueued, on a transfer stream of its own, into the slot
//     whose previous reader was N+2 deliveries back; the transfer stream
//     waits for that reader's release event and records the slot's ready
//     event, which the attention waits for (items 2 and 3: two slots of
//     margin, deliveries issued after enqueue, recycling ordered stream to
//     stream, never through the host);
//  3. depth N (0 = ordered path exactly) and the budget: (N+2) slots must fit
//     the budget, checked before anything is allocated on every plan, a
//     declined ring is latched, and the transfer stream is created with the
//     ring and released with it (section Device memory).
// The ordered path delivers a layer in stream order on the caller's stream
// into one buffer, then attends.  Both paths attend over the same rows with
// the same chunking, so their outputs are byte-identical.
#include "ctx.h"

#include <algorithm>
#include <chrono>
#include <cstring>
#include <thread>

namespace kvc {

int cuda_fail(Ctx *c, cudaError_t e, const char *what);
int dev_alloc(Ctx *c, void **p, int64_t bytes, const char *what);
void dev_free(Ctx *c, void *p, int64_t bytes);

#define KVC_CU(c, call)                                                                                            \
    do {                                                                                                           \
        cudaError_t e_ = (call);                                                                                   \
        if (e_ != cudaSuccess) return cuda_fail((c), e_, #call);                                                   \
    } while (0)

// ------------------------------------------------------ split-K planning ----

// Split-K plan of one launch: rows per chunk and the kernel configuration.
// Rows per chunk: enough chunks that every SM gets work in whole waves, no
// chunk longer than ATTN_MAX_CHUNK_ROWS (few long chunks amortise each CTA's
// prologue and merge: one wave of long chunks beats several of short ones),
// at least 64 rows (partials stay a small fraction of the bytes read).
// Configuration 1 (two CTAs per SM, q8_0) takes over when the work exceeds
// one wave of configuration 0 at the longest chunks: measured, it streams such
// long contexts faster, and below that it is slower.  Depends only on the row
// counts, the sequence count, the geometry and the SM count.
struct ChunkPlan {
    int C;                   // rows per chunk (the longest, with per-sequence lengths)
    int cfg;
    std::vector<int32_t> Cs; // per-sequence rows per chunk (a batch of a symmetric cache), else empty
};

// Per-sequence chunk lengths for a batch: every sequence is cut into equal
// chunks (a multiple of 16 rows), so no sequence ends in a short chunk.  CTAs
// of nearly equal length run in lockstep waves, so for k = 1, 2, ... waves the
// smallest target length whose chunks fill at most k whole waves is found,
// and the plan with the least k * (longest chunk + a per-wave cost in rows) is
// kept; the per-wave cost stands for a CTA's prologue and merges (about 5 us:
// 800 rows for one CTA per SM, 400 for two).  Measured on the 32-sequence
// batch of lengths U[1024, 32768]: three whole waves of 4816-row chunks run
// in 0.204 ms against 0.224 ms for one uniform length, and a length that
// leaves a partial wave (2016 rows: 0.222 ms) loses the gain.
static void batch_plan(const Ctx *c, int n_seq, const int32_t *rows, ChunkPlan &pl, int64_t slots, int cap) {
    const int64_t cmax = ATTN_MAX_CHUNK_ROWS;
    const int64_t ovh = pl.cfg ? 400 : 800;
    auto len_of = [](int64_t n, int64_t C) {
        const int64_t ch = std::max<int64_t>(1, (n + C - 1) / C);
        int64_t len = (((n + ch - 1) / ch) + 15) / 16 * 16;
        // at least 64 rows (or the whole sequence), at most C
        len = std::min<int64_t>(C, std::max<int64_t>(len, std::min<int64_t>(64, (n + 15) / 16 * 16)));
        return std::max<int64_t>(len, 16);
    };
    auto ctas_at = [&](int64_t C) {
        int64_t t = 0;
        for (int i = 0; i < n_seq; ++i) {
            const int64_t n = rows[i];
            t += std::max<int64_t>(1, (n + len_of(n, C) - 1) / len_of(n, C));
        }
        return t * c->Hk;
    };
    // the longest sequence needs at most `cap` chunks
    int64_t cmin = 64;
    for (int i = 0; i < n_seq; ++i) cmin = std::max<int64_t>(cmin, ((int64_t)rows[i] + cap - 1) / cap);
    cmin = (cmin + 15) / 16 * 16;
    if (cmin > cmax) return; // keep the uniform plan
    double best = -1.0;
    int64_t best_C = 0;
    const int64_t min_waves = std::max<int64_t>(1, (ctas_at(cmax) + slots - 1) / slots);
    for (int64_t k = min_waves; k <= min_waves + 3; ++k) {
        // smallest C (multiple of 16 in [cmin, cmax]) whose chunks fill at most k waves
        int64_t lo = cmin / 16, hi = cmax / 16;
        if (ctas_at(hi * 16) > k * slots) continue;
        while (lo < hi) {
            const int64_t mid = (lo + hi) / 2;
            if (ctas_at(mid * 16) <= k * slots) hi = mid;
            else lo = mid + 1;
        }
        const int64_t C = lo * 16;
        int64_t longest = 0;
        for (int i = 0; i < n_seq; ++i) longest = std::max(longest, std::min<int64_t>(len_of(rows[i], C), rows[i]));
        const double t = (double)k * (double)(longest + ovh);
        if (best < 0 || t < best) {
            best = t;
            best_C = C;
        }
    }
    if (best < 0) return;
    pl.Cs.resize((size_t)n_seq);
    int64_t longest = 0;
    for (int i = 0; i < n_seq; ++i) {
        pl.Cs[(size_t)i] = (int32_t)len_of(rows[i], best_C);
        longest = std::max<int64_t>(longest, pl.Cs[(size_t)i]);
    }
    pl.C = (int)std::max<int64_t>(longest, 64);
}

static ChunkPlan chunk_plan(const Ctx *c, int n_seq, const int32_t *rows) {
    int64_t total = 0;
    for (int i = 0; i < n_seq; ++i) total += rows[i];
    const int64_t work = std::max<int64_t>(total * c->Hk, 1);
    const int64_t cmax = ATTN_MAX_CHUNK_ROWS;
    ChunkPlan pl;
    pl.cfg = (c->occ2 > 0 && work > (int64_t)c->sms * c->occ * cmax) ? 1 : 0;
    int64_t C;
    if (c->chunk_override) {
        C = c->chunk_override;
    } else {
        int64_t slots = (int64_t)c->sms * (pl.cfg ? c->occ2 : c->occ);
        // One CTA per SM and short chunks: leave as many SMs as the previous launch has last
        // CTAs (one per sequence and KV head, still merging its partials when this launch
        // starts), so that no CTA of this launch starts late behind them and holds up its
        // merge.  Measured: 16k 16.0 -> 14.4 us; with long chunks the lost SMs cost more.
        const int64_t busy = (int64_t)n_seq * c->Hk;
        if (!pl.cfg && busy * 8 <= slots && work <= (slots - busy) * 4096) slots -= busy;
        const int64_t waves = std::max<int64_t>(1, (work + slots * cmax - 1) / (slots * cmax));
        C = (work + waves * slots - 1) / (waves * slots);
        C = std::min<int64_t>(cmax, std::max<int64_t>(64, (C + 15) / 16 * 16));
        if (n_seq == 1 && rows[0] > 0) {
            // One sequence: the same number of chunks (or fewer), each a whole number of
            // 128-row tiles, so that a chunk's tiles start on tile boundaries of the pages
            // instead of leaving a fragment tile at each end.  Measured on 64-layer graphs:
            // 4k 8.43 -> 7.65 us, 16k 14.3 -> 13.3 us, 64k 33.6 -> 32.0 us.
            const int64_t k = (rows[0] + C - 1) / C;
            const int64_t c2 = ((rows[0] + k - 1) / k + 127) / 128 * 128;
            if (c2 <= cmax) C = c2;
        }
    }
    // at most `cap` chunks per (sequence, kv head)
    const int cap = attn_merge_cap(c->tk, c->D, c->r, pl.cfg);
    for (int i = 0; i < n_seq; ++i) {
        const int64_t need = ((int64_t)rows[i] + cap - 1) / cap;
        if (need > C) C = (need + 15) / 16 * 16;
    }
    pl.C = (int)std::min<int64_t>(C, cmax);
    if (n_seq > 1 && !c->chunk_override && c->tv == c->tk) {
        int64_t slots = (int64_t)c->sms * (pl.cfg ? c->occ2 : c->occ);
        const int64_t busy = (int64_t)n_seq * c->Hk;
        if (!pl.cfg && busy * 8 <= slots && work <= (slots - busy) * 4096) slots -= busy;
        batch_plan(c, n_seq, rows, pl, slots, cap);
    }
    return pl;
}

static int chunk_rows_plan(const Ctx *c, int n_seq, const int32_t *rows) {
    return chunk_plan(c, n_seq, rows).C;
}

} // namespace kvc

extern "C" int kvc_debug_chunk_plan(int type, int head_dim, int n_head, int n_head_kv, int sms, int occ, int occ2,
                                    int n_seq, const int32_t *rows, int32_t *chunk_rows, int32_t *cfg) {
    using namespace kvc;
    if (!rows || !chunk_rows || !cfg || n_seq < 1 || sms < 1 || occ < 1 || occ2 < 0) return KVC_EINVAL;
    if (type != KVC_Q8_0 && type != KVC_F16) return KVC_EINVAL;
    if (head_dim != 64 && head_dim != 128) return KVC_EINVAL;
    if (n_head_kv < 1 || n_head < 1 || n_head % n_head_kv || n_head / n_head_kv > MAX_GROUP) return KVC_EINVAL;
    if (type == KVC_F16 && occ2 != 0) return KVC_EINVAL; // f16 has one configuration
    for (int i = 0; i < n_seq; ++i)
        if (rows[i] < 0) return KVC_EINVAL;
    Ctx c;
    c.tk = c.tv = type;
    c.D = head_dim;
    c.Hk = n_head_kv;
    c.r = n_head / n_head_kv;
    c.sms = sms;
    c.occ = occ;
    c.occ2 = occ2;
    const ChunkPlan pl = chunk_plan(&c, n_seq, rows);
    *chunk_rows = pl.C;
    *cfg = pl.cfg;
    return KVC_OK;
}

extern "C" int kvc_debug_chunk_plan_seq(int type, int head_dim, int n_head, int n_head_kv, int sms, int occ,
                                        int occ2, int n_seq, const int32_t *rows, int32_t *chunk_rows_seq,
                                        int32_t *cfg) {
    using namespace kvc;
    int32_t C = 0;
    int rc = kvc_debug_chunk_plan(type, head_dim, n_head, n_head_kv, sms, occ, occ2, n_seq, rows, &C, cfg);
    if (rc) return rc;
    if (!chunk_rows_seq) return KVC_EINVAL;
    Ctx c;
    c.tk = c.tv = type;
    c.D = head_dim;
    c.Hk = n_head_kv;
    c.r = n_head / n_head_kv;
    c.sms = sms;
    c.occ = occ;
    c.occ2 = occ2;
    const ChunkPlan pl = chunk_plan(&c, n_seq, rows);
    for (int i = 0; i < n_seq; ++i) chunk_rows_seq[i] = pl.Cs.empty() ? pl.C : pl.Cs[(size_t)i];
    return KVC_OK;
}

namespace kvc {

static int grow_partials(Ctx *c, int64_t need, cudaStream_t st) {
    if (need <= c->part_floats) return KVC_OK;
    // grows only for forced chunk sizes or unusual batches (not inside graph capture)
    KVC_CU(c, cudaStreamSynchronize(st));
    dev_free(c, c->part, c->part_floats * 4);
    c->part = nullptr;
    c->part_floats = 0;
    int rc = dev_alloc(c, (void **)&c->part, need * 4, "partials");
    if (rc) return rc;
    c->part_floats = need;
    return KVC_OK;
}

int launch_attention(Ctx *c, const LayerView &lv, const CUtensorMap *tmk, const CUtensorMap *tmv, int P,
                     int64_t scale_limit, int n_seq, const AttnSeq *seqs_in, const float *q, float *out,
                     float kq_scale, cudaStream_t st, const float *app_k, const float *app_v) {
    std::vector<int32_t> rows((size_t)n_seq);
    for (int i = 0; i < n_seq; ++i) rows[(size_t)i] = seqs_in[i].n_rows;
    const ChunkPlan pl = chunk_plan(c, n_seq, rows.data());
    const int C = pl.C;
    const int64_t pf = (int64_t)attn_partial_floats(c->r, c->D);
    for (int base = 0; base < n_seq; base += MAX_SEQ_PER_LAUNCH) {
        const int cnt = std::min(MAX_SEQ_PER_LAUNCH, n_seq - base);
        AttnParams p;
        std::memset(&p, 0, sizeof(p));
        p.H = c->H;
        p.Hk = c->Hk;
        p.D = c->D;
        p.r = c->r;
        p.P = P;
        p.chunk_rows = C;
        p.n_seq = cnt;
        p.kq_scale_log2 = (float)((double)kq_scale * 1.4426950408889634);
        p.q = q;
        p.out = out;
        p.ks = lv.k.scales;
        p.vs = lv.v.scales;
        p.tickets = c->tickets;
        p.err = c->err_dev;
        p.scale_limit_bytes = scale_limit;
        // the tensor maps cover one slot (Hk x P rows) on the host paths, the layer's pool otherwise
        p.map_rows = c->host ? (int64_t)c->Hk * P : c->pool_rows;
        p.app_k = app_k;
        p.app_v = app_v;
        p.app_heads = c->Hk;
        p.app_lv = lv;
        int32_t chunks = 0;
        for (int i = 0; i < cnt; ++i) {
            AttnSeq a = seqs_in[base + i];
            const int Ci = pl.Cs.empty() ? C : pl.Cs[(size_t)(base + i)];
            a.chunk_rows = Ci;
            a.chunk0 = chunks;
            a.n_chunks = std::max(1, (a.n_rows + Ci - 1) / Ci);
            a.part0 = a.part_first = chunks;
            a.ticket = i;
            p.seq[i] = a;
            chunks += a.n_chunks;
        }
        p.total_chunks = chunks;
        if (cnt == 1) p.chunk_rows = p.seq[0].chunk_rows; // one sequence: the plain instance reads the launch's
        int rc = grow_partials(c, (int64_t)chunks * c->Hk * pf, st);
        if (rc) return rc;
        p.part = c->part;
        p.part_cap = c->part_floats;
        for (int i = 0; i < cnt; ++i) p.seq[i].pt_len = c->host ? 1 : c->max_pages;
        cudaError_t e = launch_attn(c->tk, c->tv, p, tmk, tmv, st, false, pl.cfg);
        if (e != cudaSuccess) return cuda_fail(c, e, "attention kernel");
    }
    return KVC_OK;
}

// ------------------------------------------------------- host transport ----

static int64_t slot_bytes_for(const Ctx *c, int64_t cap) {
    return (int64_t)c->Hk * cap * (c->krow + c->vrow + c->ksb + c->vsb) + 4 * 64;
}

// Capacity of a slot for a context of n rows: n rounded up to 1024 rows,
// within the host store's capacity.
static int32_t cap_for(const Ctx *c, int64_t n) {
    int64_t cap = (std::max<int64_t>(n, 1) + 1023) / 1024 * 1024;
    return (int32_t)std::min<int64_t>(cap, c->P);
}

static void free_slot(Ctx *c, Slot &s) {
    if (s.kdata) dev_free(c, s.kdata, 0);
    if (s.vdata) dev_free(c, s.vdata, 0);
    if (s.kscales) dev_free(c, s.kscales, 0);
    if (s.vscales) dev_free(c, s.vscales, 0);
    c->device_bytes -= s.bytes;
    if (s.ready) cudaEventDestroy(s.ready);
    if (s.release) cudaEventDestroy(s.release);
    s = Slot();
}

// Allocate and zero a slot.  The zeroing runs on `st`; the slot's ready
// event is recorded after it, so a delivery issued on any other stream (the
// non-blocking transfer stream) waits for it instead of racing it.
static int alloc_slot(Ctx *c, Slot &s, int32_t cap, cudaStream_t st) {
    s = Slot();
    const int64_t rows = (int64_t)c->Hk * cap;
    int rc;
    const int64_t before = c->device_bytes;
    if ((rc = dev_alloc(c, &s.kdata, rows * c->krow + 64, "slot K"))) return rc;
    if ((rc = dev_alloc(c, &s.vdata, rows * c->vrow + 64, "slot V"))) return rc;
    if (c->ksb && (rc = dev_alloc(c, (void **)&s.kscales, rows * c->ksb + 64, "slot K scales"))) return rc;
    if (c->vsb && (rc = dev_alloc(c, (void **)&s.vscales, rows * c->vsb + 64, "slot V scales"))) return rc;
    // device_bytes is adjusted by free_slot with s.bytes
    s.bytes = c->device_bytes - before;
    c->device_bytes = before + s.bytes;
    s.scale_bytes = c->ksb ? rows * c->ksb + 64 : 0;
    s.cap = cap;
    KVC_CU(c, cudaMemsetAsync(s.kdata, 0, (size_t)(rows * c->krow + 64), st));
    KVC_CU(c, cudaMemsetAsync(s.vdata, 0, (size_t)(rows * c->vrow + 64), st));
    if (s.kscales) KVC_CU(c, cudaMemsetAsync(s.kscales, 0, (size_t)(rows * c->ksb + 64), st));
    if (s.vscales) KVC_CU(c, cudaMemsetAsync(s.vscales, 0, (size_t)(rows * c->vsb + 64), st));
    std::string why;
    for (int b = 0; b < 2; ++b) {
        const int box = b ? (int)std::min<int64_t>(TMA_BIG_ROWS, rows) : TMA_BOX_ROWS;
        if (!encode_rows_map(&s.tmk[b], s.kdata, rows, c->krow, c->tk, true, &why, box) ||
            !encode_rows_map(&s.tmv[b], s.vdata, rows, c->vrow, c->tv, true, &why, box))
            return c->fail(KVC_ECUDA, why);
    }
    KVC_CU(c, cudaEventCreateWithFlags(&s.ready, cudaEventDisableTiming));
    KVC_CU(c, cudaEventCreateWithFlags(&s.release, cudaEventDisableTiming));
    KVC_CU(c, cudaEventRecord(s.ready, st));
    s.delivered = true; // holds no layer (layer -1), but a copy into it must follow the zeroing
    s.ready_stream = st;
    return KVC_OK;
}

void transport_release(Ctx *c) {
    for (auto &s : c->tr.ring) free_slot(c, s);
    c->tr.ring.clear();
    c->tr.rolling = false;
    if (c->tr.xfer) {
        cudaStreamDestroy(c->tr.xfer);
        c->tr.xfer = nullptr;
    }
    c->tr.cursor = 0;
    std::fill(c->tr.app_waited.begin(), c->tr.app_waited.end(), -1); // a new transfer stream waits afresh
}

static void dev_free_slot_memory(Ctx *c, Slot &s) {
    // free_slot without touching the bookkeeping of device_bytes twice
    free_slot(c, s);
}

// Tile slots of the rolling mode (one tile delivered ahead).
constexpr int ROLLING_SLOTS = 3;

// Bytes of one row of every KV head (K and V codes and scales).
static int64_t row_bytes_all(const Ctx *c) { return (int64_t)c->Hk * (c->krow + c->vrow + c->ksb + c->vsb); }

// Rows of a rolling tile for a layer attended over `rows` rows: whole chunks
// of that attention's chunk plan, as many as a tile slot holds.
static int32_t tile_rows_for(const Ctx *c, int32_t rows) {
    const int C = chunk_rows_plan(c, 1, &rows);
    const int32_t cap = c->tr.ring.empty() ? 0 : c->tr.ring[0].cap;
    return std::max(C, (cap / C) * C); // cap >= C when rolling is engaged
}

// Decide ordered / pipelined / rolling for a context of n rows; allocate or
// regrow the ring when it fits the budget.  *engaged: the ring is in use
// (c->tr.rolling tells whether it holds whole layers or tiles).
static int plan(Ctx *c, int64_t n, cudaStream_t st, bool *engaged) {
    *engaged = false;
    Transport &t = c->tr;
    if (t.depth == 0 || t.latched) return KVC_OK;
    auto drop_ring = [&]() -> int {
        if (!t.ring.empty()) {
            KVC_CU(c, cudaStreamSynchronize(st));
            if (t.xfer) KVC_CU(c, cudaStreamSynchronize(t.xfer));
            transport_release(c);
        }
        return KVC_OK;
    };
    auto make_ring = [&](int32_t cap, bool rolling, int slots) -> int {
        t.ring.resize((size_t)slots);
        for (auto &s : t.ring) {
            int rc = alloc_slot(c, s, cap, st);
            if (rc) {
                transport_release(c);
                return rc;
            }
        }
        KVC_CU(c, cudaStreamCreateWithFlags(&t.xfer, cudaStreamNonBlocking));
        t.cursor = 0;
        t.rolling = rolling;
        return KVC_OK;
    };
    int rc;
    const int32_t cap = cap_for(c, n);
    const int64_t need = (int64_t)(t.depth + 2) * slot_bytes_for(c, cap);
    if (need <= t.budget) {
        // whole layers
        if (t.ring.empty() || t.rolling || t.ring[0].cap < n) {
            if ((rc = drop_ring())) return rc;
            if ((rc = make_ring(cap, false, t.depth + 2))) return rc;
        }
        *engaged = true;
        return KVC_OK;
    }
    // Rolling: the ring holds tiles of a layer ("F5 - Advanced KV Cache
    // Techniques", Rolling KV: tiles streamed through a small ring, merged
    // with the online-softmax partials).  Three tile slots (one tile ahead,
    // whatever the depth): each tile costs a fixed number of API calls and
    // launches, so the budget goes into tile size rather than look-ahead;
    // each slot is a whole number of 1024-row blocks.
    const int64_t tcap = (t.budget / ROLLING_SLOTS - 4 * 64) / row_bytes_all(c) / 1024 * 1024;
    const int32_t rows = (int32_t)std::min<int64_t>(n, INT32_MAX);
    if (tcap < 1024 || tcap < chunk_rows_plan(c, 1, &rows)) {
        // declined before anything is allocated, and latched: the context only grows
        if ((rc = drop_ring())) return rc;
        t.latched = true;
        return KVC_OK;
    }
    if (t.ring.empty() || !t.rolling || t.ring[0].cap != tcap) {
        if ((rc = drop_ring())) return rc;
        if ((rc = make_ring((int32_t)tcap, true, ROLLING_SLOTS))) return rc;
    }
    *engaged = true;
    return KVC_OK;
}

// ------------------------------------------------------------- tracing ----

// Start a trace record on stream `st` (-1 when tracing is off or full).
static int trace_begin(Ctx *c, int kind, int layer, cudaStream_t st) {
    Trace &t = c->trace;
    if (!t.on || (int)t.recs.size() >= t.cap) return -1;
    const int i = (int)t.recs.size();
    if (cudaEventRecord(t.pool[2 * (size_t)i], st) != cudaSuccess) {
        cudaGetLastError();
        t.on = false;
        return -1;
    }
    t.recs.push_back(TraceRec{kind, layer, 0});
    return i;
}

static void trace_end(Ctx *c, int i, int64_t bytes, cudaStream_t st) {
    Trace &t = c->trace;
    if (i < 0) return;
    t.recs[(size_t)i].bytes = bytes;
    if (cudaEventRecord(t.pool[2 * (size_t)i + 1], st) != cudaSuccess) {
        cudaGetLastError();
        t.recs.resize((size_t)i); // drop the unfinished record
        t.on = false;
    }
}

// Issue H2D copies of rows [r0, r0 + rows) of `layer` from the host store
// into slot s (slot row 0 = layer row r0), after the slot's previous delivery
// and its previous reader.
static int deliver_range(Ctx *c, Slot &s, int layer, int32_t r0, int32_t rows, int tile, cudaStream_t x) {
    const int64_t hcap = c->P;
    if (s.delivered && s.ready_stream != x) KVC_CU(c, cudaStreamWaitEvent(x, s.ready, 0));
    if (s.consumed_once) KVC_CU(c, cudaStreamWaitEvent(x, s.release, 0));
    struct Part {
        uint8_t *host;
        void *dev;
        int rowb;
    } parts[4] = {{c->hk, s.kdata, c->krow}, {c->hv, s.vdata, c->vrow}, {c->hks, s.kscales, c->ksb},
                  {c->hvs, s.vscales, c->vsb}};
    const int ti = trace_begin(c, 0, layer, x);
    int64_t moved = 0;
    for (auto &pt : parts) {
        if (!pt.rowb || rows == 0) continue;
        const uint8_t *src = pt.host + ((int64_t)layer * c->Hk * hcap + r0) * pt.rowb;
        KVC_CU(c, cudaMemcpy2DAsync(pt.dev, (size_t)s.cap * pt.rowb, src, (size_t)hcap * pt.rowb,
                                    (size_t)rows * pt.rowb, (size_t)c->Hk, cudaMemcpyHostToDevice, x));
        moved += (int64_t)rows * pt.rowb * c->Hk;
    }
    c->tr.bytes += moved;
    trace_end(c, ti, moved, x);
    s.layer = layer;
    s.r0 = r0;
    s.rows = rows;
    s.tile = tile;
    KVC_CU(c, cudaEventRecord(s.ready, x));
    s.delivered = true;
    s.ready_stream = x;
    return KVC_OK;
}

static int deliver(Ctx *c, Slot &s, int layer, int32_t rows, cudaStream_t x) {
    return deliver_range(c, s, layer, 0, rows, -1, x);
}

static Slot *find_slot(Ctx *c, int layer, int32_t rows) {
    for (auto &s : c->tr.ring)
        if (s.layer == layer && s.tile < 0 && s.rows == rows) return &s;
    return nullptr;
}

// Rolling mode: the slot holding tile `tile` of `layer` from row r0 with
// `rows` rows present.
static Slot *find_tile(Ctx *c, int layer, int tile, int32_t r0, int32_t rows) {
    for (auto &s : c->tr.ring)
        if (s.layer == layer && s.tile == tile && s.r0 == r0 && s.rows == rows) return &s;
    return nullptr;
}

static Slot &next_slot(Ctx *c) {
    Transport &t = c->tr;
    Slot &s = t.ring[(size_t)(t.cursor % (int64_t)t.ring.size())];
    ++t.cursor;
    return s;
}

// Early delivery into the next ring slot on the transfer stream.
static int deliver_early(Ctx *c, int layer) {
    Transport &t = c->tr;
    const int32_t rows = c->seqs[0].lfill[(size_t)layer];
    if (rows == 0 || find_slot(c, layer, rows)) return KVC_OK;
    if (rows > t.ring[0].cap) return KVC_OK; // the next plan grows the ring
    Slot &s = next_slot(c);
    // the host rows being delivered were written by append kernels on the compute stream
    KVC_CU(c, cudaStreamWaitEvent(t.xfer, c->app_ev[(size_t)layer], 0));
    int rc = deliver(c, s, layer, rows, t.xfer);
    if (rc) return rc;
    ++t.early;
    return KVC_OK;
}

// Rolling mode: rows the attention of `layer` will cover when it comes next
// (this step for layers not yet attended, the next step for the others; one
// token per step), and tile `tile`'s stable rows [r0, r0 + n) held now.
static int deliver_tile_early(Ctx *c, int layer, int tile, int32_t att_rows) {
    Transport &t = c->tr;
    const int32_t TR = tile_rows_for(c, att_rows);
    const int32_t r0 = tile * TR;
    const int32_t held = c->seqs[0].lfill[(size_t)layer];
    const int32_t n = std::min(held, std::min(att_rows, r0 + TR)) - r0;
    if (n <= 0 || find_tile(c, layer, tile, r0, n)) return KVC_OK;
    Slot &s = next_slot(c);
    if (t.app_waited[(size_t)layer] != c->app_gen[(size_t)layer]) {
        // rows of this layer were appended since the transfer stream last waited
        KVC_CU(c, cudaStreamWaitEvent(t.xfer, c->app_ev[(size_t)layer], 0));
        t.app_waited[(size_t)layer] = c->app_gen[(size_t)layer];
    }
    int rc = deliver_range(c, s, layer, r0, n, tile, t.xfer);
    if (rc) return rc;
    ++t.early;
    ++t.tiles;
    return KVC_OK;
}

static void slot_layer_view(const Slot &s, LayerView &lv) {
    lv.k.data = s.kdata;
    lv.k.scales = reinterpret_cast<uint16_t *>(s.kscales);
    lv.v.data = s.vdata;
    lv.v.scales = reinterpret_cast<uint16_t *>(s.vscales);
}

int transport_append(Ctx *c, int layer, int n_tok, const float *k, const float *v, int in_heads, cudaStream_t st) {
    Seq &q = c->seqs[0];
    const int32_t fill = q.lfill[(size_t)layer];
    AppendDst d[2];
    int nd = 1;
    const int64_t lo = (int64_t)layer * c->Hk * c->P;
    d[0].lv.k.data = c->hk_d + lo * c->krow;
    d[0].lv.k.scales = c->ksb ? reinterpret_cast<uint16_t *>(c->hks_d + lo * c->ksb) : nullptr;
    d[0].lv.v.data = c->hv_d + lo * c->vrow;
    d[0].lv.v.scales = c->vsb ? reinterpret_cast<uint16_t *>(c->hvs_d + lo * c->vsb) : nullptr;
    d[0].pt = nullptr;
    d[0].off = 0;
    d[0].row0 = fill;
    d[0].P = c->P;
    // rows written this step also go straight into the slot holding the
    // layer's stable prefix (rolling mode: the tile they fall in), after that
    // delivery has landed
    Slot *s = nullptr;
    if (c->tr.rolling && !c->tr.ring.empty()) {
        const int32_t TR = tile_rows_for(c, fill + n_tok);
        const int tile = fill / TR;
        s = find_tile(c, layer, tile, tile * TR, fill - tile * TR);
        if (s && fill + n_tok > s->r0 + std::min(TR, s->cap)) s = nullptr;
    } else {
        s = find_slot(c, layer, fill);
        if (s && fill + n_tok > s->cap) s = nullptr;
    }
    if (s) {
        KVC_CU(c, cudaStreamWaitEvent(st, s->ready, 0));
        slot_layer_view(*s, d[1].lv);
        d[1].pt = nullptr;
        d[1].off = 0;
        d[1].row0 = fill - s->r0;
        d[1].P = s->cap;
        nd = 2;
    }
    cudaError_t e = launch_append(c->tk, c->tv, c->Hk, in_heads, c->D, n_tok, k, v, d, nd, st);
    if (e != cudaSuccess) return cuda_fail(c, e, "append kernel");
    KVC_CU(c, cudaEventRecord(c->app_ev[(size_t)layer], st));
    ++c->app_gen[(size_t)layer];
    if (nd == 2) s->rows = fill + n_tok - s->r0;
    return KVC_OK;
}

// Rolling mode: attention of `layer` over its tiles, each one launch writing
// its chunks' partials at their place in the whole layer's chunk plan; the
// ticket counts every chunk of the layer, so the last CTA of the last tile
// merges them in chunk order.  The chunking is the ordered path's, so the
// result is the same bytes.
static int rolling_attn(Ctx *c, int layer, const float *q, float *out, float kq_scale, cudaStream_t st) {
    Transport &t = c->tr;
    Seq &sq = c->seqs[0];
    const int32_t rows = sq.lfill[(size_t)layer];
    const ChunkPlan pl = chunk_plan(c, 1, &rows);
    const int C = pl.C;
    const int32_t TR = tile_rows_for(c, rows);
    const int n_tiles = std::max(1, (rows + TR - 1) / TR);
    const int total = std::max(1, (rows + C - 1) / C);
    int rc = grow_partials(c, (int64_t)total * c->Hk * (int64_t)attn_partial_floats(c->r, c->D), st);
    if (rc) return rc;
    const int32_t recent = c->recent[0][(size_t)layer];
    for (int tile = 0; tile < n_tiles; ++tile) {
        const int32_t r0 = tile * TR, n = std::min(rows, r0 + TR) - r0;
        Slot *s = find_tile(c, layer, tile, r0, n);
        if (!s) {
            // not delivered ahead: deliver now, in stream order, into the next slot
            s = &next_slot(c);
            if ((rc = deliver_range(c, *s, layer, r0, n, tile, st))) return rc;
            ++t.in_order;
            ++t.tiles;
        }
        KVC_CU(c, cudaStreamWaitEvent(st, s->ready, 0));
        AttnParams p;
        std::memset(&p, 0, sizeof(p));
        p.H = c->H;
        p.Hk = c->Hk;
        p.D = c->D;
        p.r = c->r;
        p.P = s->cap;
        p.chunk_rows = C;
        p.n_seq = 1;
        p.kq_scale_log2 = (float)((double)kq_scale * 1.4426950408889634);
        p.q = q;
        p.out = out;
        p.ks = reinterpret_cast<uint16_t *>(s->kscales);
        p.vs = reinterpret_cast<uint16_t *>(s->vscales);
        p.tickets = c->tickets;
        p.err = c->err_dev;
        p.scale_limit_bytes = s->scale_bytes;
        p.map_rows = (int64_t)c->Hk * s->cap;
        p.part = c->part;
        p.part_cap = c->part_floats;
        AttnSeq &a = p.seq[0];
        a.page_table = c->zero_pt;
        a.off = 0;
        a.n_rows = n;
        a.chunk0 = 0;
        a.n_chunks = total;
        a.out_row = 0;
        a.ticket = 0;
        a.stable_rows = std::max(0, std::min(n, rows - recent - r0));
        a.part0 = r0 / C;
        a.part_first = 0;
        a.pt_len = 1;
        p.total_chunks = (n + C - 1) / C;
        const int ti = trace_begin(c, 1, layer, st);
        cudaError_t e = launch_attn(c->tk, c->tv, p, s->tmk, s->tmv, st, false, pl.cfg);
        if (e != cudaSuccess) return cuda_fail(c, e, "attention kernel");
        trace_end(c, ti, (int64_t)n * row_bytes_all(c), st);
        KVC_CU(c, cudaEventRecord(s->release, st));
        s->consumed_once = true;
        // look-ahead: the next tile(s), on into the following layers
        int l2 = layer, t2 = tile;
        int32_t rows2 = rows;
        for (int k = 0; k < ROLLING_SLOTS - 2; ++k) {
            if (++t2 >= std::max(1, (rows2 + tile_rows_for(c, rows2) - 1) / tile_rows_for(c, rows2))) {
                l2 = (l2 + 1) % c->L;
                t2 = 0;
                // layers after this one in the step hold sq.n rows once appended; the
                // ones before it come round again in the next step with one more row
                rows2 = l2 > layer ? sq.n : sq.n + 1;
            }
            if ((rc = deliver_tile_early(c, l2, t2, rows2))) return rc;
        }
    }
    c->clear_recent();
    return KVC_OK;
}

int transport_attn(Ctx *c, int layer, const float *q, float *out, float kq_scale, cudaStream_t st) {
    Seq &sq = c->seqs[0];
    const int32_t rows = sq.lfill[(size_t)layer];
    bool engaged = false;
    int rc = plan(c, sq.n, st, &engaged);
    if (rc) return rc;
    if (engaged && c->tr.rolling) return rolling_attn(c, layer, q, out, kq_scale, st);
    Slot *s = nullptr;
    if (engaged) {
        s = find_slot(c, layer, rows);
        if (!s) {
            // not delivered ahead: deliver now, in stream order, into the next slot
            s = &next_slot(c);
            if ((rc = deliver(c, *s, layer, rows, st))) return rc;
            ++c->tr.in_order;
        }
        KVC_CU(c, cudaStreamWaitEvent(st, s->ready, 0));
    } else {
        Slot &o = c->tr.ordered;
        if (o.cap < rows || !o.kdata) {
            if (o.kdata) {
                KVC_CU(c, cudaStreamSynchronize(st));
                dev_free_slot_memory(c, o);
            }
            if ((rc = alloc_slot(c, o, cap_for(c, std::max<int64_t>(rows, sq.n)), st))) return rc;
        }
        if ((rc = deliver(c, o, layer, rows, st))) return rc;
        ++c->tr.in_order;
        s = &o;
    }
    LayerView lv;
    slot_layer_view(*s, lv);
    AttnSeq a;
    std::memset(&a, 0, sizeof(a));
    a.page_table = c->zero_pt;
    a.off = 0;
    a.n_rows = rows;
    a.out_row = 0;
    a.stable_rows = std::max(0, rows - c->recent[0][(size_t)layer]);
    const int ti = trace_begin(c, 1, layer, st);
    rc = launch_attention(c, lv, s->tmk, s->tmv, s->cap, s->scale_bytes, 1, &a, q, out, kq_scale, st, nullptr,
                          nullptr);
    if (rc) return rc;
    trace_end(c, ti, (int64_t)rows * row_bytes_all(c), st);
    c->clear_recent();
    if (engaged) {
        KVC_CU(c, cudaEventRecord(s->release, st));
        s->consumed_once = true;
        // look-ahead: the next N layers (wrapping into the next step)
        for (int k = 1; k <= c->tr.depth; ++k) {
            if ((rc = deliver_early(c, (layer + k) % c->L))) return rc;
        }
    }
    return KVC_OK;
}

} // namespace kvc

// ------------------------------------------------------------- tracing API --
using namespace kvc;

static Ctx *trace_ctx(kvc_ctx *cc) {
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    if (!c) return nullptr;
    if (c->split) return c->part_host; // the transport belongs to the host half
    return c->host ? c : nullptr;
}

extern "C" int kvc_trace_start(kvc_ctx *cc, int max_records) {
    Ctx *c = trace_ctx(cc);
    if (!c) return cc ? reinterpret_cast<Ctx *>(cc)->fail(KVC_EINVAL, "tracing needs a host-resident or split context")
                      : KVC_EINVAL;
    if (max_records < 1 || max_records > (1 << 16)) return c->fail(KVC_EINVAL, "max_records must be in [1, 65536]");
    KVC_CU(c, cudaSetDevice(c->dev));
    Trace &t = c->trace;
    while ((int)t.pool.size() < 2 * max_records) {
        cudaEvent_t e;
        KVC_CU(c, cudaEventCreate(&e));
        t.pool.push_back(e);
    }
    t.cap = max_records;
    t.recs.clear();
    t.on = true;
    return KVC_OK;
}

extern "C" int kvc_trace_stop(kvc_ctx *cc) {
    Ctx *c = trace_ctx(cc);
    if (!c) return KVC_EINVAL;
    c->trace.on = false;
    return KVC_OK;
}

extern "C" int kvc_trace_read(kvc_ctx *cc, kvc_trace_event *out, int cap, int *n) {
    Ctx *c = trace_ctx(cc);
    if (!c) return KVC_EINVAL;
    if (!n || cap < 0 || (cap > 0 && !out)) return c->fail(KVC_EINVAL, "bad output arguments");
    Trace &t = c->trace;
    *n = (int)t.recs.size();
    if (t.recs.empty() || cap == 0) return KVC_OK;
    KVC_CU(c, cudaSetDevice(c->dev));
    // every recorded event must have completed (bounded host wait)
    const size_t last = 2 * t.recs.size();
    for (size_t i = 0; i < last; ++i) {
        const auto t0 = std::chrono::steady_clock::now();
        for (;;) {
            const cudaError_t q = cudaEventQuery(t.pool[i]);
            if (q == cudaSuccess) break;
            if (q != cudaErrorNotReady) return cuda_fail(c, q, "trace event");
            if (std::chrono::steady_clock::now() - t0 > std::chrono::milliseconds(c->timeout_ms))
                return c->fail(KVC_ETIMEDOUT, "trace events did not complete");
            std::this_thread::sleep_for(std::chrono::microseconds(50));
        }
    }
    const int m = std::min(cap, (int)t.recs.size());
    for (int i = 0; i < m; ++i) {
        float a = 0.f, b = 0.f;
        KVC_CU(c, cudaEventElapsedTime(&a, t.pool[0], t.pool[2 * (size_t)i]));
        KVC_CU(c, cudaEventElapsedTime(&b, t.pool[0], t.pool[2 * (size_t)i + 1]));
        out[i].kind = t.recs[(size_t)i].kind;
        out[i].layer = t.recs[(size_t)i].layer;
        out[i].bytes = t.recs[(size_t)i].bytes;
        out[i].t0_us = 1000.0 * a;
        out[i].t1_us = 1000.0 * b;
    }
    return KVC_OK;
}
