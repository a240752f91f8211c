// kvc_internal.h - shared declarations of the CUDA library (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "kvc.h" // include/ is on the include path

namespace kvc {

constexpr int QK = 32;                 // elements per q8_0 block
// q8_0 code bytes in device pools, host stores and staging slots are offset
// binary: the byte holds code + 128 (the int8 code with its top bit flipped),
// which the attention kernel turns into fp16 without a separate flip.  The
// state format and the no-alloc entry point's caller buffers carry plain int8
// codes; copies between the two flip the top bit of every code byte.
constexpr uint32_t CODE_FLIP = 0x80808080u;
constexpr int MAX_SEQ_PER_LAUNCH = 64; // sequences carried in one attention launch
constexpr int MAX_GROUP = 8;           // query heads per KV head supported by the attention kernel
constexpr int TMA_BOX_ROWS = 16;       // rows per small TMA box
constexpr int TMA_BIG_ROWS = 128;      // rows per large TMA box

// Device error word bits (kernels set them instead of trapping).
constexpr uint32_t ERR_WAIT_TIMEOUT = 1u << 0;
constexpr uint32_t ERR_BAD_INDEX = 1u << 1;
constexpr uint32_t ERR_BAD_CONFIG = 1u << 2;
constexpr uint32_t ERR_BAD_PAGE = 1u << 3; // attention: a page-table entry outside the tensor maps
constexpr uint32_t ERR_BAD_PART = 1u << 4; // attention: a split-K partial outside the partial buffer

// Addressing of one layer's K or V store.  Row index of (page, kv head g,
// cell) is (page * Hk + g) * P + cell; data rows are `row_bytes` long,
// q8_0 scale rows are `scale_bytes` long (fp16 per 32 elements).
struct TensorView {
    void *data;        // int8 codes (q8_0) or fp16 halves (f16)
    uint16_t *scales;  // q8_0 only, else nullptr
};

struct LayerView {
    TensorView k, v;
};

// Per-sequence description in an attention launch.
struct AttnSeq {
    const int32_t *page_table; // device, logical page -> physical page
    int32_t off;               // offset of logical row 0 in the first page
    int32_t n_rows;            // rows to attend over
    int32_t chunk0;            // first global chunk index of this sequence
    int32_t n_chunks;          // chunks of this sequence (>= 1)
    int32_t out_row;           // index of this sequence in q / out
    int32_t ticket;            // index of this sequence's ticket row
    int32_t stable_rows;       // leading rows no possibly in-flight kernel writes (readable before
                               // the programmatic-dependency wait)
    int32_t part0;             // partial slot of this launch's first chunk of the sequence
    int32_t part_first;        // partial slot of the sequence's chunk 0 (n_chunks slots from there
                               // are merged); a sequence's chunks may span several launches, the
                               // ticket counting all of them
    int32_t pt_len;            // entries of page_table
    int32_t app_row;           // row this launch quantises and stores itself (fused append), or -1
    int32_t chunk_rows;        // rows per chunk of this sequence (launches of more than one sequence)
};

struct AttnParams {
    int32_t H, Hk, D, r, P;
    int32_t chunk_rows;
    int32_t n_seq;
    int32_t total_chunks;
    float kq_scale_log2; // kq_scale * log2(e)
    const float *q;
    float *out;
    const uint16_t *ks; // K scales of this layer (q8_0), else nullptr
    const uint16_t *vs; // V scales of this layer (q8_0), else nullptr
    float *part;        // split-K partials
    int32_t *tickets;   // [MAX_SEQ_PER_LAUNCH * Hk] arrival counters, self-resetting
    uint32_t *err;      // device error word
    int64_t scale_limit_bytes; // bytes readable from ks / vs (bounds of the bulk copies)
    int64_t map_rows;          // rows the K / V tensor maps cover (pages must lie inside)
    int64_t part_cap;          // floats of the partial buffer
    // Fused quantise-on-append (the decode step): for each sequence with
    // app_row >= 0, the CTA whose chunk holds that row quantises it from
    // app_k / app_v (fp32 [.][app_heads][D], the sequence's token at index
    // out_row) into app_lv, then reads it like any other row.  app_k == nullptr: none.
    const float *app_k, *app_v;
    int32_t app_heads;
    LayerView app_lv;
    AttnSeq seq[MAX_SEQ_PER_LAUNCH];
};

// Launch the decode attention kernel for one layer.  tmk / tmv each point at
// a pair of maps over the same rows: boxes of TMA_BOX_ROWS rows, then of
// TMA_BIG_ROWS rows.
// raw_codes: q8_0 codes are plain int8 (caller buffers) instead of offset binary.
// cfg 0: one CTA per SM; cfg 1 (q8_0 only): two CTAs per SM, for launches whose
// work exceeds one wave of cfg 0 at the longest chunks.
// type: the K type; type_v: the V type (the same, or KVC_Q4_0 with q8_0 K,
// head_dim 128 and configuration 0).
cudaError_t launch_attn(int type, int type_v, const AttnParams &p, const CUtensorMap *tmk, const CUtensorMap *tmv,
                        cudaStream_t st, bool raw_codes = false, int cfg = 0);
int attn_ctas_per_sm(int type, int D, int r, int cfg = 0); // 0: the configuration does not exist
int attn_merge_cap(int type, int D, int r, int cfg = 0);   // most chunks per (sequence, kv head) a launch may use
constexpr int ATTN_MAX_CHUNK_ROWS = 8000;                  // a chunk spans at most 512 tiles
size_t attn_partial_floats(int r, int D); // floats per (chunk, kv head) partial
// Group size of the kernel instance a launch with group size r runs (partials,
// merge capacity and occupancy follow that instance): plain int8 q8_0 codes run
// the one instance for groups of up to 8.
int attn_instance_r(int type, int r, bool raw_codes);
constexpr int MAX_DEVICES = 64; // devices whose per-device state the library caches
// A process-unique id of the current CUDA context (0 if it cannot be read):
// state that belongs to a context is cached under it, so a reset device or
// another context is set up again.
uint64_t current_context_id();

// Quantise-on-append.  Destination of token t: logical row row0 + t of a
// sequence with page table pt and first-page offset off (pt == nullptr:
// single page 0, cell = row0 + t).
struct AppendDst {
    LayerView lv;
    const int32_t *pt;
    int32_t off;
    int32_t row0;
    int32_t P;
};
// k / v hold in_heads head-rows per token; the first Hk of them are stored.
cudaError_t launch_append(int type_k, int type_v, int Hk, int in_heads, int D, int n_tok, const float *k,
                          const float *v, const AppendDst *dst, int n_dst, cudaStream_t st);

// Write page-table entries: pt[idx[i]] = val[i], up to 32 per launch.
cudaError_t launch_pt_update(int32_t *pt, int n, const int32_t *idx, const int32_t *val, cudaStream_t st);

// Range copies of the sequence operations.  A run is n consecutive physical
// rows of one KV head starting at pool row `row0` (layer 0); `other` is the
// first row on the other side: a pool row (pool to pool) or the row index
// g * N + i of the packed state layout (N rows exported, g the KV head).
// Every run is applied to layers [l0, l0 + n_layers) and to each present
// tensor (K codes, V codes, K scales, V scales).
struct RowRun {
    int64_t row0;
    int64_t other;
    int32_t n;
    int32_t pad;
};
struct RunCopyArgs {
    uint8_t *base[4];    // K codes, V codes, K scales, V scales (null: absent)
    int32_t rowb[4];     // bytes per row of each
    int64_t pool_rows;   // rows of one layer pool
    uint8_t *payload;    // null: pool to pool (row0 -> other)
    int64_t layer_bytes; // payload bytes of one layer
    int64_t toff[4];     // offset of each tensor inside a payload layer
    int32_t to_payload;  // payload copies: 1 pool -> payload, 0 payload -> pool
    uint32_t flip[4];    // XOR applied to every 4 bytes copied (offset-binary <-> int8 codes)
    int32_t l0;          // first layer
    int64_t payload_rows; // rows of each tensor section of a payload layer (Hk x rows)
    uint32_t *err;        // device error word: a run outside its buffers is reported and skipped
};
cudaError_t launch_copy_runs(const RunCopyArgs &a, const RowRun *runs_dev, int64_t n_runs, int n_layers,
                             cudaStream_t st);

// RoPE shift of stored K rows.  A span is `n` consecutive physical rows
// starting at row0 = (page * Hk + g) * P + cell of the layer-0 pool; every
// span is applied to each of the n_layer layers (layer_rows apart).  cs:
// (cos, sin) of delta * theta_i for i < D/2, copied into the launch.
struct RopeSpan {
    int64_t row0;
    int32_t n;
    int32_t pad;
};
constexpr int ROPE_SPAN_MAX = 512; // rows of one span (one CTA)
cudaError_t launch_rope_shift(int type_k, int D, int mode, void *kdata, uint16_t *kscales, int64_t layer_rows,
                              int n_layer, const RopeSpan *spans_dev, int64_t n_spans, const float2 *cs,
                              uint32_t *err, cudaStream_t st);

// KeyDiff scan over one layer's K of one sequence (k_keydiff.cu).
// A block of n <= block_rows consecutive rows of one page: row0 is head
// 0's layer-0 row of the first, i0 the first row's index in the output.
struct KeyDiffBlock {
    int64_t row0;
    int32_t n;
    int32_t i0;
};
// Rows per block for a K type / head count / head size (the score kernel's
// stages must fit in shared memory), and blocks per pass-1 slice.
int keydiff_block_rows(bool q8, int Hk, int D);
int keydiff_slice_blocks();
struct KeyDiffArgs {
    bool q8;                   // K type q8_0 (offset-binary codes + fp16 scales) or f16
    int32_t Hk, D, P;          // P: rows per page (head g's row = head 0's row + g * P)
    const uint8_t *kdata;      // K pool base (codes or halves)
    const uint16_t *kscales;   // q8_0 scales (else null)
    int64_t layer_off;         // first row of the layer in the pool
    const KeyDiffBlock *blocks; // the sequence's rows
    int32_t n_blocks;
    int32_t block_rows;
    int32_t n_slices;          // pass 1: every head's blocks in slices of keydiff_slice_blocks()
    int64_t n_rows;
    float *slice_sum;          // work: [Hk][n_slices][D]
    float *mean;               // work: [Hk][D]
    float *mean_norm;          // work: [Hk]
    float *score;              // out: [n_rows], by the blocks' i0
    uint32_t *err;             // device error word (ERR_WAIT_TIMEOUT)
};
cudaError_t launch_keydiff(const KeyDiffArgs &a, int sms, cudaStream_t st);

// Encode a 2D tiled tensor map (rows x row_bytes) for the attention kernel.
bool encode_rows_map(CUtensorMap *m, const void *base, int64_t rows, int row_bytes, int type, bool swizzle,
                     std::string *why, int box_rows = TMA_BOX_ROWS);

} // namespace kvc
