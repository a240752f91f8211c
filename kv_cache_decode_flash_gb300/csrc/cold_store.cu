// cold_store.cu - host-RAM cold store of evicted KV blocks (host code).
//
// "Plan: lossless long context - derived hot/cold sizing (#5) + host-RAM KV
// cold store (#3)", section llama - KV-byte offload: a range evicted from the
// hot cache is copied into a scratch sequence, exported as state bytes and
// kept in host RAM under the range's token hash with its cache class; the
// range is then removed and the later rows slide down.  Admitting imports the
// bytes into the scratch sequence, shifts them to the tail, copies them into
// the sequence and drops the scratch (append mode).  The store is bounded in
// tokens and, when full, drops the most evictable class first and the least
// recently stored block within a class.
#include "ctx.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstring>
#include <new>
#include <string>
#include <vector>

namespace {

struct ColdBlock {
    uint64_t key = 0;
    int32_t cls = 0;
    int32_t n_tok = 0;
    int32_t first_pos = 0; // position of the block's first row when it was evicted
    uint64_t stamp = 0;    // store order (least recently stored = smallest)
    uint8_t *bytes = nullptr; // pinned host memory
    size_t size = 0;
    size_t cap = 0;           // its allocated size
};

struct ColdStore {
    int64_t budget = 0;
    int64_t tokens = 0;
    int64_t bytes = 0;
    uint64_t clock = 0;
    std::vector<ColdBlock> blocks;
    // freed pinned buffers kept for reuse (pinning host memory costs far more than filling it)
    std::vector<std::pair<uint8_t *, size_t>> spare;
    int64_t stored = 0, rejected = 0, dropped = 0, hits = 0, misses = 0;
    // restore cost model: sums over the timed admits (rows, microseconds) for a
    // least-squares line, or a model the caller set
    int64_t samples = 0;
    double sx = 0.0, sy = 0.0, sxx = 0.0, sxy = 0.0;
    bool model_set = false;
    double set_fixed = 0.0, set_per_tok = 0.0;
    std::string err;

    // The restore model: set by the caller, else fitted to the timed admits
    // (two or more distinct sizes: least squares; one size: proportional).
    // False without either.
    bool model(double *fixed, double *per_tok) const {
        if (model_set) {
            *fixed = set_fixed;
            *per_tok = set_per_tok;
            return true;
        }
        if (samples == 0) return false;
        const double n = (double)samples, den = n * sxx - sx * sx;
        if (samples >= 2 && den > 1e-9 * n * sxx) {
            *per_tok = (n * sxy - sx * sy) / den;
            *fixed = (sy - *per_tok * sx) / n;
        } else {
            *fixed = 0.0;
            *per_tok = sy / sx;
        }
        return true;
    }
    static constexpr size_t MAX_SPARE = 4;

    // A pinned buffer of at least `size` bytes (the smallest spare that fits, else a new one);
    // *cap is its allocated size.
    uint8_t *take(size_t size, size_t *cap) {
        int best = -1;
        for (size_t i = 0; i < spare.size(); ++i)
            if (spare[i].second >= size && (best < 0 || spare[i].second < spare[(size_t)best].second)) best = (int)i;
        if (best >= 0) {
            uint8_t *p = spare[(size_t)best].first;
            *cap = spare[(size_t)best].second;
            spare.erase(spare.begin() + best);
            return p;
        }
        uint8_t *p = nullptr;
        if (cudaMallocHost(&p, size) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        *cap = size;
        return p;
    }
    void give(uint8_t *p, size_t cap) {
        if (!p) return;
        if (spare.size() < MAX_SPARE) {
            spare.emplace_back(p, cap);
        } else {
            cudaFreeHost(p);
        }
    }

    int fail(int code, const std::string &m) {
        err = m;
        return code;
    }
    int find(uint64_t key) const {
        for (size_t i = 0; i < blocks.size(); ++i)
            if (blocks[i].key == key) return (int)i;
        return -1;
    }
    void drop(int i) {
        ColdBlock &b = blocks[(size_t)i];
        give(b.bytes, b.cap);
        tokens -= b.n_tok;
        bytes -= (int64_t)b.size;
        blocks.erase(blocks.begin() + i);
    }
    // Blocks to drop so that n more tokens of class cls fit, in drop order:
    // among blocks at least as evictable as cls, the most evictable class
    // first, the least recently stored first within a class.  False when they
    // cannot make room (the new block is then not kept).
    bool victims(int64_t n, int32_t cls, std::vector<uint64_t> &out) const {
        out.clear();
        if (n > budget) return false;
        std::vector<const ColdBlock *> cand;
        for (auto &b : blocks)
            if (b.cls >= cls) cand.push_back(&b);
        std::sort(cand.begin(), cand.end(), [](const ColdBlock *a, const ColdBlock *b) {
            return a->cls != b->cls ? a->cls > b->cls : a->stamp < b->stamp;
        });
        int64_t used = tokens;
        for (const ColdBlock *b : cand) {
            if (used + n <= budget) break;
            out.push_back(b->key);
            used -= b->n_tok;
        }
        return used + n <= budget;
    }
};

ColdStore *S(kvc_cold *s) { return reinterpret_cast<ColdStore *>(s); }
const ColdStore *S(const kvc_cold *s) { return reinterpret_cast<const ColdStore *>(s); }

// Rows of sequence q with positions in [p0, p1), and the smallest such position.
int64_t rows_in(const kvc::Seq &q, int64_t p0, int64_t p1, int32_t *first) {
    int64_t n = 0;
    int32_t lo = INT32_MAX;
    for (int32_t p : q.pos)
        if (p >= p0 && p < p1) {
            ++n;
            lo = std::min(lo, p);
        }
    *first = n ? lo : 0;
    return n;
}

} // namespace

using kvc::Ctx;

extern "C" {

int kvc_cold_create(int64_t budget_tokens, kvc_cold **out) {
    if (!out) return KVC_EINVAL;
    *out = nullptr;
    if (budget_tokens < 1) return KVC_EINVAL;
    ColdStore *s = new (std::nothrow) ColdStore();
    if (!s) return KVC_ENOMEM;
    s->budget = budget_tokens;
    *out = reinterpret_cast<kvc_cold *>(s);
    return KVC_OK;
}

void kvc_cold_destroy(kvc_cold *cs) {
    if (!cs) return;
    ColdStore *s = S(cs);
    while (!s->blocks.empty()) s->drop((int)s->blocks.size() - 1);
    for (auto &sp : s->spare) cudaFreeHost(sp.first);
    delete s;
}

const char *kvc_cold_last_error(const kvc_cold *cs) {
    return cs ? S(cs)->err.c_str() : "null store";
}

int kvc_cold_evict(kvc_ctx *cc, kvc_cold *cs, int seq, int scratch, int p0, int p1, uint64_t key, int cls,
                   int *stored, int32_t *n_tok) {
    if (!cc || !cs || !stored || !n_tok) return KVC_EINVAL;
    ColdStore *s = S(cs);
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    *stored = 0;
    *n_tok = 0;
    if (c->host) return s->fail(KVC_EINVAL, "the cold store needs a device-resident context");
    const int n_seq = (int)c->seqs.size();
    if (seq < 0 || seq >= n_seq || scratch < 0 || scratch >= n_seq || seq == scratch)
        return s->fail(KVC_EINVAL, "bad sequence or scratch id");
    if (p0 < 0 || p1 <= p0 || cls < 0) return s->fail(KVC_EINVAL, "bad range or class");
    if (c->seqs[(size_t)scratch].n != 0) return s->fail(KVC_EINVAL, "the scratch sequence is not empty");
    int32_t first = 0;
    const int64_t n = rows_in(c->seqs[(size_t)seq], p0, p1, &first);
    *n_tok = (int32_t)n;
    if (n == 0) return KVC_OK;
    // decide first, so that a block that will not be kept is not exported
    const int old = s->find(key);
    if (old >= 0) s->drop(old);
    std::vector<uint64_t> vict;
    const bool keep = s->victims(n, cls, vict);
    int rc;
    if (keep) {
        if ((rc = kvc_seq_cp(cc, seq, scratch, p0, p1))) return s->fail(rc, "seq_cp into the scratch sequence");
        size_t size = 0;
        if ((rc = kvc_state_get(cc, scratch, -1, -1, nullptr, 0, &size))) {
            kvc_seq_rm(cc, scratch, -1, -1);
            return s->fail(rc, "state size");
        }
        size_t cap = 0;
        uint8_t *buf = s->take(size, &cap);
        if (!buf) {
            kvc_seq_rm(cc, scratch, -1, -1);
            return s->fail(KVC_ENOMEM, "pinned host memory for a cold block");
        }
        size_t got = 0;
        rc = kvc_state_get(cc, scratch, -1, -1, buf, size, &got);
        int rc2 = kvc_seq_rm(cc, scratch, -1, -1);
        if (rc || rc2) {
            s->give(buf, cap);
            return s->fail(rc ? rc : rc2, "exporting the block");
        }
        for (uint64_t k : vict) {
            s->drop(s->find(k));
            ++s->dropped;
        }
        ColdBlock b;
        b.key = key;
        b.cls = cls;
        b.n_tok = (int32_t)n;
        b.first_pos = first;
        b.stamp = ++s->clock;
        b.bytes = buf;
        b.size = got;
        b.cap = cap;
        s->blocks.push_back(b);
        s->tokens += n;
        s->bytes += (int64_t)got;
        ++s->stored;
        *stored = 1;
    } else {
        ++s->rejected;
    }
    // the range leaves the hot cache either way: remove it and slide the rest down
    if ((rc = kvc_seq_rm(cc, seq, p0, p1))) return s->fail(rc, "seq_rm of the evicted range");
    if ((rc = kvc_seq_add(cc, seq, p1, -1, -(p1 - p0)))) return s->fail(rc, "sliding the later rows");
    return KVC_OK;
}

int kvc_cold_admit(kvc_ctx *cc, kvc_cold *cs, int seq, int scratch, uint64_t key, int *hit, int32_t *n_tok) {
    if (!cc || !cs || !hit || !n_tok) return KVC_EINVAL;
    ColdStore *s = S(cs);
    Ctx *c = reinterpret_cast<Ctx *>(cc);
    *hit = 0;
    *n_tok = 0;
    if (c->host) return s->fail(KVC_EINVAL, "the cold store needs a device-resident context");
    const int n_seq = (int)c->seqs.size();
    if (seq < 0 || seq >= n_seq || scratch < 0 || scratch >= n_seq || seq == scratch)
        return s->fail(KVC_EINVAL, "bad sequence or scratch id");
    if (c->seqs[(size_t)scratch].n != 0) return s->fail(KVC_EINVAL, "the scratch sequence is not empty");
    const int i = s->find(key);
    if (i < 0) {
        ++s->misses;
        return KVC_OK;
    }
    const ColdBlock b = s->blocks[(size_t)i];
    int64_t tail = 0;
    for (int32_t p : c->seqs[(size_t)seq].pos) tail = std::max<int64_t>(tail, (int64_t)p + 1);
    size_t used = 0;
    const auto t0 = std::chrono::steady_clock::now();
    int rc = kvc_state_set(cc, scratch, b.bytes, b.size, &used);
    if (!rc && tail != b.first_pos) rc = kvc_seq_add(cc, scratch, -1, -1, (int)(tail - b.first_pos));
    if (!rc) rc = kvc_seq_cp(cc, scratch, seq, -1, -1);
    const int rc2 = kvc_seq_rm(cc, scratch, -1, -1);
    if (rc || rc2) return s->fail(rc ? rc : rc2, "importing the block");
    // the restore's cost (every call above is synchronous): one sample of the model
    const double us = std::chrono::duration<double, std::micro>(std::chrono::steady_clock::now() - t0).count();
    const double x = (double)b.n_tok;
    ++s->samples;
    s->sx += x;
    s->sy += us;
    s->sxx += x * x;
    s->sxy += x * us;
    s->drop(i);
    ++s->hits;
    *hit = 1;
    *n_tok = b.n_tok;
    return KVC_OK;
}

int kvc_cold_find(const kvc_cold *cs, uint64_t key, int32_t *n_tok, int32_t *cls) {
    if (!cs || !n_tok || !cls) return KVC_EINVAL;
    const ColdStore *s = S(cs);
    const int i = s->find(key);
    *n_tok = i < 0 ? 0 : s->blocks[(size_t)i].n_tok;
    *cls = i < 0 ? -1 : s->blocks[(size_t)i].cls;
    return KVC_OK;
}

int kvc_cold_restore_model(const kvc_cold *cs, double *fixed_us, double *per_token_us, int64_t *samples) {
    if (!cs || !fixed_us || !per_token_us || !samples) return KVC_EINVAL;
    const ColdStore *s = S(cs);
    *samples = s->samples;
    if (!s->model(fixed_us, per_token_us)) {
        *fixed_us = 0.0;
        *per_token_us = 0.0;
    }
    return KVC_OK;
}

int kvc_cold_set_restore_model(kvc_cold *cs, double fixed_us, double per_token_us) {
    if (!cs) return KVC_EINVAL;
    ColdStore *s = S(cs);
    if (per_token_us < 0.0) { // back to the fitted model
        s->model_set = false;
        return KVC_OK;
    }
    if (!(fixed_us >= 0.0) || !std::isfinite(fixed_us) || !std::isfinite(per_token_us))
        return s->fail(KVC_EINVAL, "the model needs finite fixed_us >= 0 and per_token_us >= 0");
    s->model_set = true;
    s->set_fixed = fixed_us;
    s->set_per_tok = per_token_us;
    return KVC_OK;
}

int kvc_cold_plan_admit(const kvc_cold *cs, uint64_t key, double recompute_fixed_us, double recompute_us_per_token,
                        int *restore, double *restore_us, int32_t *n_tok) {
    if (!cs || !restore || !restore_us || !n_tok) return KVC_EINVAL;
    if (!std::isfinite(recompute_fixed_us) || !std::isfinite(recompute_us_per_token)) return KVC_EINVAL;
    const ColdStore *s = S(cs);
    const int i = s->find(key);
    *restore = 0;
    *restore_us = 0.0;
    *n_tok = i < 0 ? 0 : s->blocks[(size_t)i].n_tok;
    if (i < 0) return KVC_OK; // nothing stored: recompute
    double fixed = 0.0, per_tok = 0.0;
    if (!s->model(&fixed, &per_tok)) {
        // no restore timed yet: the stored bytes are lossless and the pages' default
        *restore = 1;
        *restore_us = -1.0;
        return KVC_OK;
    }
    const double n = (double)*n_tok;
    *restore_us = fixed + per_tok * n;
    *restore = *restore_us < recompute_fixed_us + recompute_us_per_token * n ? 1 : 0;
    return KVC_OK;
}

int kvc_cold_get_stats(const kvc_cold *cs, kvc_cold_stats *o) {
    if (!cs || !o) return KVC_EINVAL;
    const ColdStore *s = S(cs);
    std::memset(o, 0, sizeof(*o));
    o->budget_tokens = s->budget;
    o->tokens = s->tokens;
    o->bytes = s->bytes;
    o->blocks = (int32_t)s->blocks.size();
    o->stored = s->stored;
    o->rejected = s->rejected;
    o->dropped = s->dropped;
    o->hits = s->hits;
    o->misses = s->misses;
    return KVC_OK;
}

} // extern "C"
