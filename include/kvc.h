/*
 * kvc.h - decode attention over a quantised grouped-query KV cache on one
 * GB300 GPU (sm_103a), with the sequence operations a host-RAM cold store is
 * built from and a host-resident mode that streams each layer's K/V from
 * pinned host memory through a staging ring.
 *
 * Sources (web pages; cited by title and section):
 *  [F5]   "F5 - Advanced KV Cache Techniques" (opencoti llamafile docs).
 *  [COLD] "Plan: lossless long context - derived hot/cold sizing (#5) +
 *          host-RAM KV cold store (#3)" (contenox modeld docs).
 *  [R4]   "sched: pipeline the delivery of a host-resident KV cache (R4)"
 *          (llama.cpp pull request).
 *
 * Conventions for every call:
 *  - Every function returns a kvc_status (0 = KVC_OK, negative = error) except
 *    kvc_destroy, kvc_last_error, kvc_status_str and kvc_params_init.  A bad
 *    argument never aborts the process; on error the call leaves the cache as
 *    it was (no partial effect) unless the status is KVC_ECUDA or
 *    KVC_EINTERNAL, after which the context should be destroyed.
 *    kvc_last_error(ctx) gives a one-line description of the last error.
 *  - Ownership: the library owns every KV byte (device pools, pinned host
 *    store, staging ring, work space).  The caller owns q, out, k, v (device
 *    pointers, e.g. torch tensors) and all host byte buffers; the library
 *    never keeps a caller pointer after a call returns.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream).  kvc_append, kvc_attn_decode and kvc_decode_step only
 *    enqueue work on it and return without waiting; calls on one context must be issued from one
 *    host thread and be ordered on the device (one stream, or events).
 *    The sequence and state operations are synchronous: they wait for all
 *    device work already issued in the process, run, and return when their
 *    effect is complete (kvc_state_get's bytes are valid at return).
 *  - A context is not thread-safe; distinct contexts are independent.
 *  - Positions are int32.  Ranges [p0, p1) are half-open; p0 < 0 means 0 and
 *    p1 < 0 means "no upper bound" (the llama.cpp sequence-op convention).
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kvc_ctx kvc_ctx;

typedef enum kvc_status {
    KVC_OK = 0,
    KVC_EINVAL = -1,     /* bad argument, unsupported geometry or call order */
    KVC_ENOMEM = -2,     /* device or pinned host allocation failed */
    KVC_ENOSPC = -3,     /* no free cells / pages left for new rows */
    KVC_ERANGE = -4,     /* position out of range (e.g. a shift below 0) */
    KVC_EFORMAT = -5,    /* state bytes malformed or of another geometry */
    KVC_ECUDA = -6,      /* a CUDA call failed (sticky errors included) */
    KVC_ETIMEDOUT = -7,  /* a bounded host wait or device wait gave up */
    KVC_EINTERNAL = -8   /* a kernel reported an inconsistency */
} kvc_status;

/* Storage type of K and of V.
 * KVC_Q8_0: blocks of 32 elements stored as 32 int8 codes plus one fp16
 * scale d; d = max|x| / 127 and code = round-half-away-from-zero(x * (1/d))
 * in fp32, scale stored as fp16(d) round-to-nearest-even.  The type is named
 * in [F5] section M6 ("-ctk q8_0") and [R4] section Measurements ("q8_0
 * K/V"); the pages give no bit layout, so this plainest reading is pinned.
 * KVC_Q4_0 (V only, with q8_0 K and head_dim 128: the asymmetric cache of
 * [F5] section M6 - PolyKV, "-ctk q8_0 -ctv q4_0"): blocks of 32 elements
 * stored as 32 four-bit codes plus one fp16 scale d.  The pages name the type
 * without defining it; the reading used: m = the element of largest
 * magnitude, sign kept (the first one on ties), d = m / -8, code =
 * min(15, trunc(x * (1/d) + 8.5)) with the product and the sum each rounded
 * to fp32, scale stored as fp16(d); value = (code - 8) * d.  Byte j of a
 * block (16 bytes) holds code j in its low four bits and code j + 16 in its
 * high four bits.
 * KVC_F16: IEEE binary16, round to nearest even. */
typedef enum kvc_type { KVC_F16 = 1, KVC_Q4_0 = 2, KVC_Q8_0 = 8 } kvc_type;

/* Where a context keeps its K/V.
 * KVC_DEVICE: device HBM, paged, any number of sequences.
 * KVC_HOST_PINNED: pinned host RAM, one sequence (id 0); each layer's rows
 * are delivered to the device through a staging ring before attention
 * ([R4] section What it does).  Only kvc_append and kvc_attn_decode are
 * available; the sequence and state operations return KVC_EINVAL.
 * KVC_SPLIT_HEADS: a per-head residency split ("F5 - Advanced KV Cache
 * Techniques", sections M2 HeadInfer and M3 NEO): KV heads 0 .. gpu_heads-1
 * (whole GQA groups: query heads 0 .. gpu_heads*H/Hk - 1) live in device HBM
 * as with KVC_DEVICE, the others in pinned host RAM as with
 * KVC_HOST_PINNED, delivered through the staging ring.  kvc_attn_decode runs
 * two attention launches on the disjoint head ranges (device heads first, so
 * they overlap the host heads' transfers) whose outputs sit side by side on
 * the head axis.  One sequence (id 0); only kvc_append, kvc_attn_decode and
 * the pipeline / introspection calls apply.
 */
typedef enum kvc_residency { KVC_DEVICE = 0, KVC_HOST_PINNED = 1, KVC_SPLIT_HEADS = 2 } kvc_residency;

/* Rotary pairing used by kvc_seq_add.  NEOX pairs (i, i + D/2); NORM pairs
 * (2i, 2i + 1).  The pages do not say which; NEOX is the default. */
typedef enum kvc_rope { KVC_ROPE_NEOX = 0, KVC_ROPE_NORM = 1 } kvc_rope;

typedef struct kvc_params {
    int32_t n_layer;    /* >= 1 */
    int32_t n_head;     /* query heads H; a multiple of n_head_kv */
    int32_t n_head_kv;  /* KV heads Hk; query head h reads KV head h / (H/Hk) */
    int32_t head_dim;   /* D: 64 or 128 */
    int32_t n_ctx;      /* device: cells per layer shared by all sequences;
                           host-resident: capacity of the one sequence */
    int32_t n_seq_max;  /* sequence ids are 0 .. n_seq_max-1 */
    int32_t type_k;     /* kvc_type: KVC_Q8_0 or KVC_F16 */
    int32_t type_v;     /* kvc_type: the same as type_k, or KVC_Q4_0 with
                           type_k KVC_Q8_0 and head_dim 128 */
    float rope_base;    /* theta_i = rope_base^(-2i/D) */
    int32_t rope_mode;  /* kvc_rope */
    int32_t residency;  /* kvc_residency */
    int32_t device;     /* CUDA device ordinal */
    int32_t page_rows;  /* device residency: cells per page, a multiple of 16
                           in [16, 4096]; 0 selects 256 */
    int32_t gpu_heads;  /* KVC_SPLIT_HEADS: KV heads kept on the device,
                           1 .. n_head_kv-1; ignored otherwise */
} kvc_params;

/* Fill *p with defaults: 1 layer, 8 heads, 2 KV heads, D 64, 512 cells,
 * 1 sequence, q8_0/q8_0, base 10000, NEOX, device residency, device 0. */
void kvc_params_init(kvc_params *p);

/* Create a context: validates *p, allocates the K/V store (device pools or
 * pinned host store), the work space and the per-sequence page tables.
 * On success *out owns them until kvc_destroy.  Errors: KVC_EINVAL
 * (geometry), KVC_ENOMEM, KVC_ECUDA. */
int kvc_create(const kvc_params *p, kvc_ctx **out);

/* Free everything the context owns (waits for its device work).  NULL is a no-op. */
void kvc_destroy(kvc_ctx *c);

const char *kvc_last_error(const kvc_ctx *c);
const char *kvc_status_str(int status);

/* Quantise-on-append: write n_tok new rows of layer `layer` for sequence
 * `seq` at positions pos0 .. pos0+n_tok-1.
 * k, v: device fp32 [n_tok][n_head_kv][head_dim], contiguous, 16-byte aligned.
 * The K/V rows of a token are written per layer, as a model produces them
 * (the cpy_k/cpy_v writes of [F5] section M2 - HeadInfer).  The first layer
 * to append a position creates the row (allocating cells); the other layers
 * must then append the same positions in the same order.
 * Host-resident contexts also write the rows into the staging slot that
 * holds this layer ([R4] section What it does, item 1: the rows written
 * this step are the ones outside the stable prefix).
 * Errors: KVC_EINVAL (ids, n_tok < 1, positions not matching the rows other
 * layers created), KVC_ENOSPC (no free pages), KVC_ECUDA. */
int kvc_append(kvc_ctx *c, int layer, int seq, int pos0, int n_tok, const float *k,
               const float *v, void *stream);

/* Single-token decode attention for n_seq sequences of one layer:
 *   out[i][h][:] = softmax_j(kq_scale * q[i][h] . K_j) V_j
 * over every row j the sequence holds for that layer, with K/V read as
 * stored (q8_0 or f16) and query head h reading KV head h / (H/Hk)
 * ([F5] sections M2/M3: grouped-query heads stay in whole KV-head groups).
 * Computed as split-K flash decoding: KV chunks of the same sequence run on
 * different CTAs and their partial (max, sum, output) triples are merged with
 * the online-softmax rule ([F5] section M4 - ScoutAttention: merge via
 * FlashAttention's online-softmax; section F5-opt W4: inter-tile online
 * softmax).  Accumulation is fp32; the merge order is fixed, so a call is
 * bitwise repeatable.
 * seq_ids: HOST int32[n_seq] (distinct ids).  q: device fp32
 * [n_seq][n_head][head_dim]; out: device fp32, same shape (may not alias q);
 * both 16-byte aligned.
 * A sequence with no rows yields a zero output row.
 * Host-resident contexts: n_seq must be 1 and seq_ids[0] 0; the layer's rows
 * are delivered through the staging ring first ([R4] section What it does).
 * Errors: KVC_EINVAL, KVC_ECUDA. */
int kvc_attn_decode(kvc_ctx *c, int layer, int n_seq, const int32_t *seq_ids, const float *q,
                    float *out, float kq_scale, void *stream);

/* One decode step of one layer for n_seq sequences: sequence seq_ids[i]
 * appends one token at position pos[i] (its K/V head-rows are row i of k / v)
 * and then attends over all its rows with query row i of q.  The result, out
 * and the stored rows, is bitwise that of kvc_append(c, layer, seq_ids[i],
 * pos[i], 1, k + i*n_head_kv*head_dim, v + ..., stream) for every i followed
 * by kvc_attn_decode(c, layer, n_seq, seq_ids, q, out, kq_scale, stream)
 * ([F5] section M2 - HeadInfer: the per-layer cpy_k/cpy_v writes, then the
 * attention over the cache; the q8_0 block of the decode-attention statement).
 * On device-resident contexts it is one launch: the CTA that attends over a
 * sequence's last chunk quantises the new row, stores it and reads it back
 * like the others, so no separate append kernel sits between the producer of
 * k/v/q and the attention.  Host-resident and split contexts take n_seq 1,
 * sequence 0, and run the two calls.
 * seq_ids, pos: HOST int32[n_seq].  k, v: device fp32 [n_seq][n_head_kv]
 * [head_dim]; q, out: device fp32 [n_seq][n_head][head_dim]; all 16-byte
 * aligned; out may not alias q.
 * Errors: as kvc_append and kvc_attn_decode; every check (ids, positions, free
 * pages) is made before anything changes, so a failed call leaves the context
 * as it was (except KVC_ECUDA). */
int kvc_decode_step(kvc_ctx *c, int layer, int n_seq, const int32_t *seq_ids, const int32_t *pos,
                    const float *k, const float *v, const float *q, float *out, float kq_scale,
                    void *stream);

/* Remove the rows of `seq` whose position is in [p0, p1), in every layer
 * (MemorySeqRemove, [COLD] section llama - KV-byte offload; the context
 * shift's discard, [F5] section M1).  Rows after the removed ones keep their
 * order; whole pages are freed, partly used boundary pages are compacted
 * on the device.  An empty range is a no-op.  Errors: KVC_EINVAL. */
int kvc_seq_rm(kvc_ctx *c, int seq, int p0, int p1);

/* Copy the rows of `src` whose position is in [p0, p1) to the end of `dst`,
 * all layers, K and V, positions unchanged (MemorySeqCopy, [COLD] section
 * llama - KV-byte offload).  The copy is physical: later operations on one
 * sequence never change the other.  src == dst is a no-op.
 * Errors: KVC_EINVAL, KVC_ENOSPC. */
int kvc_seq_cp(kvc_ctx *c, int src, int dst, int p0, int p1);

/* Add `delta` to the position of every row of `seq` whose position is in
 * [p0, p1) and rotate its stored K by delta positions (MemorySeqAdd, [COLD]
 * section llama - KV-byte offload; shifted imports rotate RoPE-positioned
 * keys by the destination/source position delta, [COLD] section OpenVINO -
 * KV-byte offload).  Each rotary pair (see kvc_rope) turns by the angle
 * delta * rope_base^(-2i/D), computed in fp64 on the host.  q8_0 K rows are
 * dequantised, rotated in fp32 and requantised; f16 rows are rotated in fp32
 * and rounded to f16.  V is untouched.  delta == 0 is a no-op.
 * Errors: KVC_EINVAL, KVC_ERANGE (a position would leave [0, INT32_MAX]). */
int kvc_seq_add(kvc_ctx *c, int seq, int p0, int p1, int delta);

/* Export the rows of `seq` with position in [p0, p1) (in row order) as bytes
 * (StateSeqGetData, [COLD] section llama - KV-byte offload: evicted KV is
 * parked in host RAM as bytes).  dst: HOST buffer of cap bytes; dst == NULL
 * only reports the size in *n_written.  Errors: KVC_EINVAL, KVC_ENOSPC when
 * cap is too small (*n_written then holds the size needed).
 *
 * Byte format, version 1, little endian; every section is zero-padded to a
 * multiple of 16 bytes:
 *   header, 64 bytes: u32 magic 0x3143564B ("KVC1"), u32 version = 1,
 *     u32 n_layer, u32 n_head_kv, u32 head_dim, u32 type_k, u32 type_v,
 *     u32 n_tok, u64 payload_bytes (everything after the positions),
 *     24 zero bytes;
 *   positions: int32 pos[n_tok];
 *   payload: for each layer, the K section then the V section, where a q8_0
 *     section is codes int8 [n_head_kv][n_tok][head_dim] followed by scales
 *     u16 (fp16 bits) [n_head_kv][n_tok][head_dim/32], a q4_0 section is
 *     packed codes u8 [n_head_kv][n_tok][head_dim/2] followed by scales as
 *     for q8_0, and an f16 section is u16 [n_head_kv][n_tok][head_dim]. */
int kvc_state_get(kvc_ctx *c, int seq, int p0, int p1, void *dst, size_t cap,
                  size_t *n_written);

/* Import bytes written by kvc_state_get into `seq`, appending the rows at
 * their stored positions (append mode: StateSeqSetData, [COLD] section
 * llama - KV-byte offload).  src: HOST buffer of n bytes.  *n_read (may be
 * NULL) receives the bytes consumed.  The header must match this context's
 * n_layer, n_head_kv, head_dim, type_k and type_v.
 * Errors: KVC_EFORMAT (bad magic, version, geometry, length), KVC_ENOSPC. */
int kvc_state_set(kvc_ctx *c, int seq, const void *src, size_t n, size_t *n_read);

/* KeyDiff distinctiveness of every row of `seq` in one layer ([F5] section
 * M1 - retention-aware context shift, which evicts the keys least
 * distinctive by cosine similarity): score_j = (1/n_head_kv) * sum over KV
 * heads g of (1 - cos(K_j,g, mu_g)), mu_g the mean of head g's keys over the
 * sequence's rows, the cosine read as 0 when either norm is 0.  Keys are
 * the stored (post-RoPE) K, q8_0 dequantised exactly; scores are fp32.
 * Rows come in position order.  scores: HOST float[cap], or NULL to only
 * receive the row count in *n.  layer < 0 selects n_layer / 2 (the page's
 * default representative layer).  Device-resident contexts only.
 * Errors: KVC_EINVAL, KVC_ENOSPC (cap below the row count). */
int kvc_seq_key_scores(kvc_ctx *c, int seq, int layer, float *scores, int32_t cap, int32_t *n);

/* Retention-aware context shift ([F5] section M1): among the windows of
 * n_discard consecutive rows (position order) that lie inside
 * [n_keep, rows - n_recent), remove the one with the smallest sum of
 * KeyDiff scores (kvc_seq_key_scores of `layer`; sums in fp64, the first
 * window on ties) with kvc_seq_rm over the positions it spans, then move
 * every later position down over the gap with kvc_seq_add (which re-rotates
 * those rows' K).  *p0 receives the first removed position, or -1 when no
 * window fits (nothing changes).  Positions are taken to be distinct.
 * Errors: KVC_EINVAL (n_discard < 1, n_keep or n_recent < 0), and those of
 * the operations it runs. */
int kvc_seq_evict_window(kvc_ctx *c, int seq, int layer, int n_keep, int n_discard, int n_recent, int32_t *p0);

/* Pipeline depth N of the host-resident transport: deliveries are issued N
 * layers ahead into an (N+2)-slot ring; 0 is the ordered path exactly
 * (deliver, then attend, in stream order).  Default 1 ([R4] section What it
 * does: --kv-pipeline-depth).  Changing it releases the ring and clears the
 * budget latch.  Device-resident contexts accept and ignore it (the
 * transport is never created).  Errors: KVC_EINVAL (n < 0 or n > 16). */
int kvc_pipeline_depth(kvc_ctx *c, int n);

/* Device-memory budget of the staging ring, in bytes.  Default 128 MiB
 * ([R4] section Device memory: --kv-pipeline-budget).  The need,
 * (N+2) * bytes of one layer's K+V over the current context, is checked
 * before anything is allocated on every plan.  A ring of whole layers that
 * does not fit falls back to rolling mode ([F5] section Rolling KV): three
 * slots (at any N >= 1) hold tiles of a layer, each the largest whole number
 * of 1024 rows that lets three fit the budget, and each layer is attended
 * tile by tile while the next tile is delivered; tiles are whole chunks of the
 * layer's split-K plan, so the output bytes equal the ordered path's.  When
 * even a 1024-row tile (or one chunk) does not fit, the ring is declined and
 * the decision is latched; the transfer stream and events are created only
 * when a ring is engaged and released with it, and a declined context runs
 * the ordered path.  Changing the budget releases the ring and clears the
 * latch.  Errors: KVC_EINVAL. */
int kvc_pipeline_budget(kvc_ctx *c, size_t bytes);

/* Number of rows `seq` holds in every layer (after all appends of a step). */
int kvc_seq_n_tokens(const kvc_ctx *c, int seq, int32_t *n);

/* Positions of the rows of `seq`, in row order.  pos: HOST int32[cap];
 * *n receives the row count (pos may be NULL to query it). */
int kvc_seq_positions(const kvc_ctx *c, int seq, int32_t *pos, int32_t cap, int32_t *n);

/* Counters describing the host-resident transport and the caches. */
typedef struct kvc_stats {
    int32_t ring_engaged;       /* 1 while a ring is allocated */
    int32_t ring_declined;      /* 1 once the budget latch tripped */
    int32_t ring_slots;         /* N+2 when engaged, else 0 */
    int32_t transfer_stream;    /* 1 while the transfer stream exists */
    int64_t slot_bytes;         /* bytes of one slot (one layer's K+V) */
    int64_t ring_bytes;         /* device bytes held by the ring */
    int64_t ordered_bytes;      /* device bytes of the ordered-path buffer */
    int64_t deliveries_early;   /* deliveries issued ahead on the transfer stream */
    int64_t deliveries_ordered; /* deliveries issued in stream order */
    int64_t bytes_delivered;    /* host-to-device bytes issued */
    int64_t pages_total;        /* device residency: pages per layer */
    int64_t pages_free;
    int64_t device_bytes;       /* all device memory held by the context */
    int64_t host_pinned_bytes;  /* pinned host memory held by the context */
    int32_t rolling;            /* 1 while the ring holds tiles of a layer (rolling mode) */
    int32_t tile_rows;          /* rows of one tile slot in rolling mode, else 0 */
    int64_t tiles_delivered;    /* rolling mode: tile deliveries issued */
} kvc_stats;

int kvc_get_stats(const kvc_ctx *c, kvc_stats *out);

/* Force the split-K chunk length in rows (a multiple of 16) for every later
 * kvc_attn_decode; 0 restores the automatic choice, which depends only on
 * the row counts, the geometry and the device's SM count.  Errors: KVC_EINVAL. */
int kvc_set_chunk_rows(kvc_ctx *c, int rows);

/* Test hook, no context and no GPU needed: the split-K plan an attention
 * launch over n_seq sequences of rows[i] rows would use, for a KV type,
 * head_dim and head counts, on a device of `sms` SMs where configuration 0
 * fits occ CTAs per SM and configuration 1 (q8_0, two CTAs of half the
 * size) occ2 (0: not available).  *chunk_rows: rows per chunk, at most 8000
 * (for one sequence, a whole number of 128-row tiles where that fits); *cfg: the
 * configuration.  rows: HOST int32[n_seq].  Errors: KVC_EINVAL. */
int kvc_debug_chunk_plan(int type, int head_dim, int n_head, int n_head_kv, int sms, int occ, int occ2,
                         int n_seq, const int32_t *rows, int32_t *chunk_rows, int32_t *cfg);

/* Test hook, no context and no GPU needed: the same plan with each
 * sequence's own rows per chunk.  A batch (n_seq > 1) of a cache whose K and
 * V types are equal cuts every sequence into equal chunks, their length
 * chosen over whole waves of chunks; a single sequence has the one length of
 * kvc_debug_chunk_plan.  chunk_rows_seq: HOST int32[n_seq].  Errors: KVC_EINVAL. */
int kvc_debug_chunk_plan_seq(int type, int head_dim, int n_head, int n_head_kv, int sms, int occ, int occ2,
                             int n_seq, const int32_t *rows, int32_t *chunk_rows_seq, int32_t *cfg);

/* Test hook, no context and no GPU needed: the rows of a sequence holding
 * positions pos[0 .. n) that the sequence operations select for the range
 * [p0, p1) (p0 < 0: from 0; p1 < 0: to the end).  linear != 0 states that the
 * positions are consecutive (pos[r] == pos[0] + r), which a context records
 * and then selects by arithmetic; a false statement is rejected.  The result
 * does not depend on linear.  pos: HOST int32[n]; rows: HOST int64[n] or NULL
 * (receives the selected rows in row order); *count: rows selected; *first:
 * the first of them (0 when none); *contiguous: 1 when they are one run of
 * consecutive rows.  Errors: KVC_EINVAL. */
int kvc_debug_select_rows(const int32_t *pos, int32_t n, int linear, int p0, int p1, int64_t *rows,
                          int64_t *count, int64_t *first, int32_t *contiguous);

/* Limit, in milliseconds, of every bounded host wait of the synchronous
 * operations (default 120000).  A wait that runs out returns KVC_ETIMEDOUT. */
int kvc_set_timeout_ms(kvc_ctx *c, int ms);

/* Host-side fault injection for tests: the next `n` internal allocations
 * succeed and the ones after fail with KVC_ENOMEM; n < 0 disables it. */
int kvc_debug_fail_alloc_after(kvc_ctx *c, int n);

/* Timeline of the host-resident transport, for measuring it (the pages show
 * the pipeline's engagement by a scheduler dump; [R4] section Measurements).
 * While tracing is on, a host-resident or split context records a timed CUDA
 * event pair around every delivery (the copies of one layer or tile, on the
 * stream that runs them: the transfer stream when pipelined, the caller's
 * stream when ordered) and around every attention launch of the transport
 * (on the caller's stream, after it has waited for the delivery).
 * kvc_trace_start: clear the records and trace the next max_records
 * (1 .. 65536) deliveries and launches; creates 2 * max_records events (kept
 * until kvc_destroy).  kvc_trace_stop: stop recording.  kvc_trace_read: wait
 * (bounded) for the recorded events, then write up to cap records into out
 * (HOST), times in microseconds from the first record's start; *n receives
 * the number recorded.  Errors: KVC_EINVAL (a device-resident context, bad
 * arguments), KVC_ETIMEDOUT, KVC_ECUDA. */
typedef struct kvc_trace_event {
    int32_t kind;  /* 0 delivery (host -> device copies), 1 attention launch */
    int32_t layer;
    int64_t bytes; /* delivery: bytes copied; attention: K/V bytes of the rows attended */
    double t0_us;  /* start (after the waits that precede it on its stream) */
    double t1_us;  /* end */
} kvc_trace_event;
int kvc_trace_start(kvc_ctx *c, int max_records);
int kvc_trace_stop(kvc_ctx *c);
int kvc_trace_read(kvc_ctx *c, kvc_trace_event *out, int cap, int *n);

/* Read and clear the device error word that kernels set instead of
 * trapping (a bounded wait that gave up, an index out of range).
 * *word receives it (0 = none).  Waits for the context's device work. */
int kvc_check_device_error(kvc_ctx *c, uint32_t *word);

/* Decode attention over caller-owned K/V that allocates no memory.
 * The pages have no counterpart for this call; it exists for callers that
 * cannot let a library call cudaMalloc: serving runtimes that reserve all
 * device memory up front and hand it out from their own arena (an
 * allocation behind their back breaks their accounting or simply fails),
 * and latency-critical paths that cannot afford an allocation's implicit
 * device synchronisation.  It computes the same thing as kvc_attn_decode
 * for one sequence of one layer, with the same kernel, without a context:
 *   out[h][:] = softmax_j(kq_scale * q[h] . K_j) V_j,  j < n_kv.
 * type: KVC_Q8_0 or KVC_F16.  K and V are the caller's device buffers, laid
 * out head-major like one layer of the state export format:
 *   q8_0: k, v = int8 codes [n_head_kv][n_kv][head_dim], ks, vs = fp16 scale
 *         bits [n_head_kv][n_kv][head_dim/32]; f16: k, v = fp16 halves
 *         [n_head_kv][n_kv][head_dim], ks = vs = NULL.
 * q, out: device fp32 [n_head][head_dim].  Every pointer 16-byte aligned;
 * scale buffers readable up to the next multiple of 16 bytes.
 * n_kv = 0 gives out = 0, as kvc_attn_decode does for an empty sequence
 * (k, v, ks and vs may then be NULL).
 * Work space (split-K partials, arrival tickets, error word) lives in one
 * fixed 8 MiB device array inside the library, which every GPU that loads
 * the library holds until the process exits.  The first call on a device
 * (and the first in a new context of it, e.g. after a device reset) does a
 * set-up with that device current: it looks up the array's device address
 * and the SM count, which allocates nothing.  Make that first call before
 * any stream capture.  All calls share the array and it keeps the previous
 * call's contents: the call clears what must start at zero in stream order,
 * and calls whose kernels overlap on the GPU (other streams, other threads)
 * race on it, so order them.
 * The kernel's own guards (a bounded wait that gave up, an index outside its
 * buffers) set a word in that work space that this call does not report:
 * there is no context whose later calls could read it.  Arguments that pass
 * the host checks below cannot trigger them.
 * Errors: KVC_EINVAL (types, shapes, null or misaligned pointers),
 * KVC_ERANGE (n_kv so large that the partials do not fit the 8 MiB work
 * space; plain kvc_attn_decode has no such limit), KVC_ECUDA. */
int kvc_attn_decode_static(int type, int n_head, int n_head_kv, int head_dim, int n_kv, const void *k,
                           const uint16_t *ks, const void *v, const uint16_t *vs, const float *q,
                           float *out, float kq_scale, void *stream);

/* ---------------------------------------------------------------------
 * Host-RAM cold store ("Plan: lossless long context", #3 Host-RAM KV cold
 * store + retrieval, llama KV-byte offload): token ranges evicted from a
 * device-resident context are kept as state bytes (kvc_state_get format) in
 * pinned host memory, keyed by a caller-supplied 64-bit token hash, so they
 * can be paged back losslessly.  The store is bounded in tokens.  When a new
 * block does not fit, blocks are dropped most evictable class first and,
 * within a class, least recently stored first; only blocks at least as
 * evictable as the new one are dropped, otherwise the new block is not kept
 * (loss happens only at the cold tier, for the most evictable classes).
 * A block lives in one tier: admitting it removes it from the store.  On a
 * miss the caller recomputes the tokens (re-prefill), the pages' fallback.
 * Not thread-safe; a store may serve several contexts of the same geometry.
 * ------------------------------------------------------------------- */
typedef struct kvc_cold kvc_cold;

typedef struct kvc_cold_stats {
    int64_t budget_tokens;
    int64_t tokens;      /* tokens held */
    int64_t bytes;       /* state bytes held (pinned host memory) */
    int32_t blocks;
    int32_t pad;
    int64_t stored;      /* evictions whose block was kept */
    int64_t rejected;    /* evictions whose block was not kept (too large, or only less
                            evictable blocks to drop) */
    int64_t dropped;     /* blocks dropped to make room */
    int64_t hits;        /* admits that found their block */
    int64_t misses;      /* admits that did not */
} kvc_cold_stats;

/* A store holding at most budget_tokens tokens (>= 1).  Errors: KVC_EINVAL, KVC_ENOMEM. */
int kvc_cold_create(int64_t budget_tokens, kvc_cold **out);
/* Free the store and its blocks.  NULL is a no-op. */
void kvc_cold_destroy(kvc_cold *s);
/* Detail of the store's last error (empty when none). */
const char *kvc_cold_last_error(const kvc_cold *s);

/* Evict the rows of `seq` with positions in [p0, p1) (p0 >= 0, p1 > p0)
 * from device-resident context c: copy them into sequence `scratch` (which
 * must be empty), export it into the store under `key` with class `cls`
 * (>= 0; larger = more evictable), drop the scratch, remove the rows from
 * `seq` and slide the later positions down by p1 - p0 (kvc_seq_cp,
 * kvc_state_get, kvc_seq_rm, kvc_seq_add).  The rows leave the context even
 * when the block is not kept: *stored tells (1 kept, 0 not).  A block
 * already stored under `key` is replaced.  *n_tok: rows evicted.
 * Errors: KVC_EINVAL (arguments, a non-empty scratch, a host-resident
 * context), the context calls' errors (c's kvc_last_error has the detail),
 * KVC_ENOMEM (pinned host memory). */
int kvc_cold_evict(kvc_ctx *c, kvc_cold *s, int seq, int scratch, int p0, int p1, uint64_t key, int cls,
                   int *stored, int32_t *n_tok);

/* Admit the block stored under `key` at the tail of `seq` (append mode):
 * import it into sequence `scratch` (empty), shift it so that its first row
 * lands at the position after the last row of `seq` (0 if empty), copy it
 * into `seq` and drop the scratch; the block leaves the store.  *hit = 1 and
 * *n_tok = its rows when found; *hit = 0 and *n_tok = 0 on a miss (nothing
 * changes).  Errors as for kvc_cold_evict; on an error the block stays in
 * the store and the scratch is emptied. */
int kvc_cold_admit(kvc_ctx *c, kvc_cold *s, int seq, int scratch, uint64_t key, int *hit, int32_t *n_tok);

/* Restore versus recompute ([COLD] #3: bulk restore of KV bytes beats
 * re-prefilling a large block, recompute wins for small ones; "restore-vs-
 * recompute latency policy").  The store keeps a cost model of restoring,
 *   restore_us(n) = fixed_us + per_token_us * n   (n rows of the block),
 * fitted by least squares to the admits it has timed (the host wall clock of
 * each kvc_cold_admit that hit: import, shift and copy, all synchronous;
 * with one block size only, a line through 0), unless the caller set one.
 * kvc_cold_restore_model: the model (zeros while there is none) and the
 * number of timed admits.  kvc_cold_set_restore_model: use the caller's
 * model (fixed_us >= 0, per_token_us >= 0); per_token_us < 0 returns to
 * the fitted one.  kvc_cold_plan_admit: for the block under `key`, *n_tok
 * its rows (0 when absent), *restore_us the model's estimate and *restore =
 * 1 when that is below the caller's cost of recomputing the block,
 * recompute_fixed_us + recompute_us_per_token * n_tok (the library runs no
 * model, so the caller supplies it).  An absent block gives *restore = 0 (recompute);
 * a present block without any model gives *restore = 1 and *restore_us = -1
 * (lossless bytes first, the pages' default).  Errors: KVC_EINVAL. */
int kvc_cold_restore_model(const kvc_cold *s, double *fixed_us, double *per_token_us, int64_t *samples);
int kvc_cold_set_restore_model(kvc_cold *s, double fixed_us, double per_token_us);
int kvc_cold_plan_admit(const kvc_cold *s, uint64_t key, double recompute_fixed_us, double recompute_us_per_token,
                        int *restore, double *restore_us, int32_t *n_tok);

/* The rows (*n_tok, 0 when absent) and class of the block under `key`. */
int kvc_cold_find(const kvc_cold *s, uint64_t key, int32_t *n_tok, int32_t *cls);
int kvc_cold_get_stats(const kvc_cold *s, kvc_cold_stats *out);

#ifdef __cplusplus
}
#endif
#endif /* KVC_H */
