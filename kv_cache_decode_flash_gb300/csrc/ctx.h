// ctx.h - the context behind the C ABI: cache manager state (host metadata),
// device pools and the host-resident transport.  Not part of the ABI.
#pragma once

#include "kvc_internal.h"

#include <algorithm>
#include <string>
#include <vector>

namespace kvc {

// Logical rows of a sequence are contiguous: logical row r lives in page
// pages[(off + r) / P] at cell (off + r) % P.  pos[r] is its position.
// lfill[l] rows of layer l have been written; a step's appends create rows
// on the first layer and fill the others, so every sequence operation
// requires lfill[l] == n for all layers.
struct Seq {
    std::vector<int32_t> pages;
    int32_t off = 0;
    int32_t n = 0;
    std::vector<int32_t> pos;
    // pos[r] == pos[0] + r for every row (consecutive positions in row
    // order), kept by every operation that changes pos; selections by
    // position range are then arithmetic
    bool linear = true;
    std::vector<int32_t> lfill;
    int32_t dev_pages = 0; // leading entries of `pages` known to match the device table
    bool synced() const {
        for (int32_t f : lfill)
            if (f != n) return false;
        return true;
    }
};

// One staging slot of the host-resident transport: one layer's K+V over the
// context, laid out [Hk][cap][row].
struct Slot {
    void *kdata = nullptr, *vdata = nullptr;
    uint16_t *kscales = nullptr, *vscales = nullptr;
    int32_t cap = 0;
    int64_t bytes = 0;
    int64_t scale_bytes = 0; // bytes of each scale buffer
    CUtensorMap tmk[2], tmv[2]; // 16-row and 128-row boxes
    cudaEvent_t ready = nullptr, release = nullptr;
    int32_t layer = -1; // layer held (-1 none)
    int32_t rows = 0;   // rows of that layer present (from row r0)
    int32_t tile = -1;  // rolling mode: tile index of the rows held, first row r0
    int32_t r0 = 0;
    bool delivered = false; // a delivery was issued into the slot (its ready event is recorded)
    cudaStream_t ready_stream = nullptr; // the stream that recorded it
    bool consumed_once = false;
};

struct Transport {
    int depth = 1;
    int64_t budget = 128ll << 20;
    bool latched = false;
    std::vector<Slot> ring; // engaged ring (depth + 2 slots) or empty
    bool rolling = false;   // ring slots hold tiles of a layer (the whole-layer ring did not fit)
    Slot ordered;           // ordered-path buffer
    cudaStream_t xfer = nullptr;
    int64_t cursor = 0;     // deliveries issued into the ring
    int64_t early = 0, in_order = 0, bytes = 0, tiles = 0;
    std::vector<int64_t> app_waited; // per layer: append generation the transfer stream has waited for
};

// Optional timeline of the host transport (kvc_trace_*): a timed event pair
// around every delivery, on the stream that copies, and around every
// attention launch, on the caller's stream, while tracing is on.
struct TraceRec {
    int32_t kind; // 0 delivery, 1 attention
    int32_t layer;
    int64_t bytes;
};
struct Trace {
    bool on = false;
    int cap = 0;                    // records the event pool holds
    std::vector<cudaEvent_t> pool;  // 2 timed events per record
    std::vector<TraceRec> recs;
};

struct Ctx {
    kvc_params prm;
    std::string err;
    int dev = 0;
    int sms = 0;
    int occ = 1;  // attention CTAs resident per SM (from the occupancy calculator), configuration 0
    int occ2 = 0; // the same for configuration 1 (two CTAs per SM; 0 where it does not exist)
    int H = 0, Hk = 0, D = 0, r = 0, L = 0, P = 0;
    int tk = 0, tv = 0;
    int krow = 0, vrow = 0, ksb = 0, vsb = 0; // data row bytes, scale row bytes (0 for f16)
    bool host = false;
    // per-head residency split: the two halves are whole contexts of their own
    bool split = false;
    int gpu_heads = 0;
    Ctx *part_dev = nullptr, *part_host = nullptr;

    // device residency
    int32_t n_pages = 0;
    int64_t pool_rows = 0; // rows per layer = n_pages * Hk * P
    std::vector<int32_t> free_pages;
    uint8_t *kdata = nullptr, *vdata = nullptr;
    uint8_t *kscales = nullptr, *vscales = nullptr;
    int64_t kdata_bytes = 0, vdata_bytes = 0, kscale_bytes = 0, vscale_bytes = 0;
    std::vector<CUtensorMap> tmk, tmv; // per layer: [2l] 16-row boxes, [2l+1] 128-row boxes
    int32_t *pt_dev = nullptr;         // [n_seq_max][max_pages]
    int32_t max_pages = 0;
    std::vector<Seq> seqs;
    // rows appended per (sequence, layer) since the last fence (an attention
    // launch or a synchronous operation); an attention launched with a
    // programmatic dependency may read every other row before it waits
    std::vector<std::vector<int32_t>> recent;
    void clear_recent() {
        for (auto &v : recent) std::fill(v.begin(), v.end(), 0);
    }

    // host residency: pinned store [L][Hk][n_ctx][row], mapped
    uint8_t *hk = nullptr, *hv = nullptr, *hks = nullptr, *hvs = nullptr;
    uint8_t *hk_d = nullptr, *hv_d = nullptr, *hks_d = nullptr, *hvs_d = nullptr; // device aliases
    int64_t host_bytes = 0;
    Transport tr;
    Trace trace;
    std::vector<cudaEvent_t> app_ev; // per layer: recorded after each append (orders early deliveries)
    std::vector<int64_t> app_gen;    // per layer: appends recorded into app_ev
    int32_t *zero_pt = nullptr;      // device page table {0} used for slots

    // attention work space
    float *part = nullptr;
    int64_t part_floats = 0;
    int32_t *tickets = nullptr;
    uint32_t *err_dev = nullptr;
    uint32_t *err_host = nullptr; // pinned copy of the error word read by synchronous operations
    int chunk_override = 0;

    // staging for sequence / state operations
    uint8_t *staging = nullptr;
    int64_t staging_bytes = 0;
    RowRun *runs_dev = nullptr;
    int64_t runs_cap = 0;
    RopeSpan *spans_dev = nullptr;
    int64_t spans_cap = 0;
    std::vector<RopeSpan> spans_host; // span list of the last shift (kept for its capacity)
    // pinned bump arena for the small host-to-device uploads of synchronous
    // operations (run and span lists, page tables); reset when the next
    // synchronous operation starts, after the device is idle
    uint8_t *up_host = nullptr;
    int64_t up_cap = 0, up_used = 0;
    std::vector<uint8_t *> up_retired; // smaller arenas that may still feed copies of this operation
    cudaStream_t st = nullptr; // internal stream of the synchronous operations
    cudaEvent_t done = nullptr;
    // state export/import: host copies of layer groups on their own stream,
    // overlapped with the pack/unpack kernels on st (created on first use)
    static constexpr int STATE_CHUNKS = 8;
    cudaStream_t st_copy = nullptr;
    cudaEvent_t st_ev[STATE_CHUNKS + 1] = {};

    int timeout_ms = 120000;
    int fail_after = -1;
    int64_t device_bytes = 0;

    int fail(int code, const std::string &msg) {
        err = msg;
        return code;
    }
};

} // namespace kvc
