/*
 * kvc.h -- C ABI of the compressed-KV decode step on one GPU (sm_103a).
 *
 * One decode step of one layer is four calls, issued in this order on one CUDA
 * stream:
 *
 *   kvc_quantize_append   write the new token's K/V: per-token INT8/INT4 codes
 *                         into the paged pool, attention sinks kept in bf16;
 *   kvc_decode_attention  single-query, GQA-aware paged attention with the
 *                         dequantisation fused into QK^T and PV, plus the H2O
 *                         heavy-hitter score accumulation;
 *   kvc_h2o_select_evict  per KV head, choose the kept set (sinks + recent
 *                         window + top-k heavy hitters, or StreamingLLM);
 *   kvc_compact_blocks    move the kept tokens into the evicted slots and give
 *                         the emptied pages back to the pool.
 *
 * kvc_decode_step runs those four for one layer in one call;
 * kvc_decode_step_overlap does the same with the eviction on a second
 * stream.  Around them:
 * kvc_prefill_attention (a fresh prompt's causal attention and the H2O scores
 * it gives), kvc_prefill_context (a prompt over sequences that hold context,
 * each query attending to the compressed cache), kvc_release_sequences (free
 * finished sequences), and the
 * options of the cache geometry: FP8 E4M3 codes and hybrid precision (the
 * last W positions kept in bf16).  Eviction modes: H2O, StreamingLLM and
 * block-granular (whole pages by mean score).
 *
 * Sources (page title, section):
 *   - "KV Cache optimization techniques" (metaphor-xennon): 1.2 per-token
 *     quantisation, 2.2 H2O, 2.4 StreamingLLM cache, 3.2 PagedAttention cache;
 *   - "Technical Report: KV Cache Compression for Text-Only Large Language
 *     Models": 1.1 attention, 3.2 INT8 quantisation with dequantisation fused
 *     into the attention kernel and sinks kept in half precision, 3.3 sliding
 *     window, 3.4 H2O eviction;
 *   - "KV cache eviction and reuse survey" (tbxsx.cn): 3.3 H2O objective,
 *     4 block manager (block-granular eviction by mean attention score);
 *   - "KV Cache optimization techniques" also: 1.3 hybrid precision, 2.3
 *     PyramidKV budgets (host side: compressed_kv_cache_kvc_gb300/budgets.py).
 *
 * Conventions shared by every call
 *   - The caller owns all device memory and the stream.  The library never
 *     allocates or frees device memory; pointers are borrowed for the call.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *     void*; NULL = legacy default stream).  Nothing synchronises except
 *     kvc_read_status, kvc_cache_reset and kvc_cache_sync_host.
 *   - Errors the host can see (bad arguments, unsupported shapes, pool
 *     exhaustion, call-order violations) are returned before anything is
 *     enqueued; the cache is then unchanged.  Errors found on the device set
 *     bits in a device status word (KVC_DEV_*), read by kvc_read_status; the
 *     kernels skip the offending access, they never trap.
 *   - Tensors are row-major and densely packed.  bf16 tensors are raw 16-bit
 *     words.  "batch" always means the contiguous slice of sequences
 *     [seq_begin, seq_begin + batch) of the cache.
 *   - A cache handle is not thread-safe; one handle per layer.
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVC_OK = 0,
  KVC_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, out-of-range value      */
  KVC_ERR_UNSUPPORTED = 2,  /* head_dim != 128, page_size != 16, bits not 4|8,
                               E4M3 codes with bits != 8, more than 8 query
                               heads per KV head                               */
  KVC_ERR_CAPACITY = 3,     /* pool or per-sequence block table would overflow
                               (the page's allocate_sequence returning False)  */
  KVC_ERR_CUDA = 4,         /* a CUDA runtime call failed                      */
  KVC_ERR_DEVICE = 5,       /* kvc_read_status found device status bits set    */
  KVC_ERR_STATE = 6         /* call order violated (compact without select)    */
} kvc_status;

/* Device status bits (kvc_read_status). */
#define KVC_DEV_OUT_OF_BLOCKS   0x1  /* free-block stack ran empty during append */
#define KVC_DEV_BAD_BLOCK_ID    0x2  /* a block-table entry outside [0, num_blocks) */
#define KVC_DEV_BAD_KEEP_MASK   0x4  /* keep mask count differs from the plan     */
#define KVC_DEV_TABLE_OVERFLOW  0x8  /* per-sequence block table overflow         */
#define KVC_DEV_STACK_OVERFLOW  0x10 /* free-block stack overflow on release      */
#define KVC_DEV_STALE_HOST      0x20 /* a sequence held more pool slots on the
                                        device than the host mirror planned for
                                        (state bytes restored without
                                        kvc_cache_sync_host): its selection and
                                        compaction were skipped                */
#define KVC_DEV_WAIT_TIMEOUT    0x40 /* a tensor-core completion wait of the
                                        prefill ran out (about a second); that
                                        CTA's outputs are missing            */
#define KVC_DEV_PREFILL_RANGE   0x80 /* a prompt value (V) entry of magnitude
                                        65536 or more, or not finite: the
                                        prefill's P.V product takes V in fp16,
                                        saturated to +-65504, so that head's
                                        prompt outputs are inexact           */

/* Geometry of one layer's cache. */
typedef struct {
  int32_t num_q_heads;        /* Hq                                             */
  int32_t num_kv_heads;       /* Hkv; Hq % Hkv == 0 and Hq / Hkv <= 8            */
  int32_t head_dim;           /* must be 128                                    */
  int32_t page_size;          /* tokens per block, must be 16                   */
  int32_t bits;               /* 8 (INT8) or 4 (INT4, two codes per byte)       */
  int32_t num_blocks;         /* physical blocks in the pool                    */
  int32_t max_batch;          /* sequences the cache holds                      */
  int32_t max_blocks_per_seq; /* block-table row length                         */
  int32_t bf16_window;        /* hybrid precision: the last W positions of each
                                 sequence are kept in bf16 (0 = off, W <= 4096);
                                 see "Hybrid precision" below                   */
  int32_t codes;              /* KVC_CODES_INT, or KVC_CODES_E4M3 (bits = 8)     */
} kvc_config;

/* Code formats.  KVC_CODES_INT: scale = amax / (2^(bits-1) - 1), integer
 * codes.  KVC_CODES_E4M3 (FP8; the pages list FP8 among their quantisation
 * strategies): scale = amax / 448 (IEEE fp32 division), code = x / scale
 * (IEEE fp32 division) rounded to FP8 E4M3, ties to even, saturating at
 * +-448; one byte per code, same layout as INT8. */
#define KVC_CODES_INT  0
#define KVC_CODES_E4M3 1

/* Hybrid precision (bf16_window = W > 0; "KV Cache optimization techniques"
 * section 1.3, HybridPrecisionKVCache: recent tokens at 16 bits, older ones
 * quantised).  The tokens at the last W positions of a sequence (after the
 * sinks) live in a bf16 ring per (sequence, KV head), slot (position - 4)
 * mod W, and attend with their exact bf16 values; a token enters the paged
 * pool, quantised as kvc_quantize_append quantises, only when it leaves the
 * window (the append that pushes it out quantises it from the ring, with the
 * H2O score it gathered there).  Pool slots therefore hold only positions
 * < P - W.  The ring tokens are always kept, so the selection requires
 * recent >= W (H2O) or window >= W (StreamingLLM), counts them inside the
 * budget or window, and chooses among the pool slots only; block-granular
 * eviction is not available with a window (KVC_ERR_UNSUPPORTED). */

/* Opaque host handle of one layer's cache (host mirror of the sequence
 * lengths, buffer offsets, launch policy). */
typedef struct kvc_cache kvc_cache;

/* Buffers carved out of the caller's state allocation (kvc_cache_buffer). */
typedef enum {
  KVC_BUF_K_CODES = 0,    /* u8  [num_blocks][Hkv][16][128*bits/8]; INT4: code
                             2i in the low nibble of byte i, two's complement */
  KVC_BUF_V_CODES = 1,    /* same layout as K                                  */
  KVC_BUF_K_SCALE = 2,    /* f32 [num_blocks][Hkv][16]  amax/127 or amax/7      */
  KVC_BUF_V_SCALE = 3,    /* f32 [num_blocks][Hkv][16]                          */
  KVC_BUF_SLOT_POS = 4,   /* i32 [num_blocks][Hkv][16]  token position per slot */
  KVC_BUF_SCORE = 5,      /* f32 [num_blocks][Hkv][16]  accumulated H2O score   */
  KVC_BUF_SINK_K = 6,     /* bf16 [max_batch][Hkv][4][128] positions 0..3       */
  KVC_BUF_SINK_V = 7,     /* bf16 [max_batch][Hkv][4][128]                      */
  KVC_BUF_SINK_SCORE = 8, /* f32 [max_batch][Hkv][4]                            */
  KVC_BUF_BLOCK_TABLE = 9,/* i32 [max_batch][max_blocks_per_seq]               */
  KVC_BUF_SEQ_SLOTS = 10, /* i32 [max_batch]  pool slots in use (non-sink tokens)*/
  KVC_BUF_SEQ_POS = 11,   /* i32 [max_batch]  positions seen (tokens appended) */
  KVC_BUF_FREE_STACK = 12,/* i32 [num_blocks] free block ids (stack)            */
  KVC_BUF_COUNTERS = 13,  /* i32 [64]: [0] free-stack top, [1] status word,
                             [2..] plan scratch                                */
  KVC_BUF_PLAN = 14,      /* i32 [max_batch][2] (slots before, slots after) of
                             the last selection                                */
  KVC_BUF_RING_K = 15,    /* bf16 [max_batch][Hkv][W][128] hybrid window;
                             slot (position - 4) mod W; empty when W = 0       */
  KVC_BUF_RING_V = 16,    /* bf16 [max_batch][Hkv][W][128]                      */
  KVC_BUF_RING_SCORE = 17,/* f32 [max_batch][Hkv][W] H2O scores of the window   */
  KVC_BUF_COUNT = 18
} kvc_buffer_id;

/* Flags of kvc_decode_attention. */
#define KVC_ATTN_ACCUM_H2O 0x1  /* add this step's probabilities to the scores */

/* Eviction modes of kvc_h2o_select_evict. */
#define KVC_EVICT_H2O       0
#define KVC_EVICT_STREAMING 1
#define KVC_EVICT_BLOCK     2  /* whole pages by mean H2O score                        */

typedef struct {
  int32_t mode;      /* KVC_EVICT_H2O, KVC_EVICT_STREAMING or KVC_EVICT_BLOCK   */
  int32_t budget;    /* H2O: tokens kept including the 4 sinks; >= 4 + recent  */
  int32_t recent;    /* H2O: recent window kept unconditionally; BLOCK: the    */
                     /* last `recent` pool slots are never evicted             */
  int32_t window;    /* StreamingLLM: recent window (sinks kept besides it)    */
  double retention;  /* BLOCK: fraction of candidate pages kept, (0, 1]        */
} kvc_evict_params;

/* ---------------------------------------------------------------- set-up -- */

/* Bytes of device memory one layer's cache state needs (all buffers above,
 * each 256-byte aligned).  Returns 0 for an invalid or unsupported config. */
size_t kvc_state_bytes(const kvc_config* cfg);

/* Create a host handle over caller-owned device memory `d_state` (at least
 * kvc_state_bytes bytes, 256-byte aligned).  Touches no GPU.  *out receives
 * the handle; release it with kvc_cache_destroy (which frees host memory only). */
kvc_status kvc_cache_create(const kvc_config* cfg, void* d_state, size_t state_bytes,
                            kvc_cache** out);
void kvc_cache_destroy(kvc_cache* cache);

/* Empty the cache: zero every buffer, fill the free-block stack with
 * `h_block_order` (host array of num_blocks distinct ids, popped from its end;
 * NULL = ascending ids) and zero the host mirror.  Synchronises `stream`. */
kvc_status kvc_cache_reset(kvc_cache* cache, const int32_t* h_block_order, void* stream);

/* Release the sequences [seq_begin, seq_begin + batch) (the paged cache's
 * free_sequence, "KV Cache optimization techniques" section 3.2): their
 * pages return to the free-block stack and their lengths become 0, so the
 * slots take a new prompt.  Idempotent: an empty sequence is left as it is.
 * One launch (none when every sequence of the slice is empty); a pending
 * selection is dropped. */
kvc_status kvc_release_sequences(kvc_cache* cache, int32_t seq_begin, int32_t batch, void* stream);

/* Device pointer and size of one buffer of the state (for inspection). */
kvc_status kvc_cache_buffer(const kvc_cache* cache, int32_t which, void** d_ptr, size_t* bytes);

/* Host mirror of one sequence: pool slots used and positions seen. */
kvc_status kvc_cache_lengths(const kvc_cache* cache, int32_t seq, int32_t* slots, int32_t* positions);

/* Reload the host mirror from the device state (after the caller restored the
 * state bytes from a snapshot).  Synchronises `stream`. */
kvc_status kvc_cache_sync_host(kvc_cache* cache, void* stream);

/* Scratch bytes kvc_decode_attention / kvc_h2o_select_evict /
 * kvc_compact_blocks need for a slice of `batch` sequences (one size fits all
 * three calls; the buffer may be reused between calls on the same stream). */
size_t kvc_workspace_bytes(const kvc_cache* cache, int32_t batch);

/* ---------------------------------------------------------------- step ---- */

/* Quantise-on-write ("KV Cache optimization techniques" 1.2; Technical Report
 * 3.2).  Appends n_new tokens to each sequence of the slice.
 *   d_k, d_v: bf16 [batch][Hkv][n_new][128] on the device, 8-byte aligned.
 * For every (token, KV head) row of K and of V: amax over the 128 values,
 * scale = amax / 127 (INT8) or amax / 7 (INT4) in IEEE fp32, code =
 * round-half-even(x / scale) (IEEE fp32 division) clamped to [-127, 127] or
 * [-8, 7]; a zero row has scale 0 and codes 0.  Tokens at positions 0..3 are
 * attention sinks: stored unchanged in bf16 and never quantised (Technical
 * Report 3.2).  New pages come from the device free-block stack; their score
 * starts at 0.  n_new == 0 is a no-op.  With KVC_CODES_E4M3 the scale is
 * amax / 448 and the codes FP8 E4M3 (see "Code formats"); with a bf16 window
 * the newest tokens go to the ring and the tokens they push out of it are
 * quantised into the pool (see "Hybrid precision").  Appends of 64 tokens or
 * more that push no window token out, from 16-byte aligned d_k and d_v, take
 * two launches, others one (the same results either way).
 * Errors: KVC_ERR_INVALID_ARG for a slice outside [0, max_batch), n_new < 0
 * or a null or misaligned pointer; KVC_ERR_CAPACITY when a sequence would
 * exceed max_blocks_per_seq pages or the pool has too few free blocks
 * (nothing is written). */
kvc_status kvc_quantize_append(kvc_cache* cache, int32_t seq_begin, int32_t batch, int32_t n_new,
                               const void* d_k, const void* d_v, void* stream);

/* Decode attention with fused dequantisation (Technical Report 1.1 and 3.2)
 * and H2O score accumulation (Technical Report 3.4).
 *   d_q:   bf16 [batch][Hq][128] one query per head, 16-byte aligned;
 *   d_out: bf16 [batch][Hq][128].
 * Query head j reads KV head j / (Hq/Hkv).  For each query head:
 *   out = softmax(sm_scale * q . k_t) . v_t over the sinks (bf16 values) and
 *   every pool slot (k_t = code * scale), accumulated in fp32.
 * With KVC_ATTN_ACCUM_H2O, every attended token's score (sinks included) grows
 * by the sum over the query heads of its KV head of its softmax probability.
 * Every sequence of the slice must hold at least one token.
 * d_workspace: kvc_workspace_bytes(cache, batch) bytes, 256-byte aligned.
 * Errors: KVC_ERR_INVALID_ARG for a slice outside the cache, a null or
 * misaligned pointer, sm_scale not positive and finite, unknown flags, a
 * short workspace or an empty sequence; KVC_ERR_UNSUPPORTED for batch >
 * 1024.  Two launches (split-K, merge with the scores), three with a bf16
 * window; the split launch is skipped when no sequence holds a pool page. */
kvc_status kvc_decode_attention(kvc_cache* cache, int32_t seq_begin, int32_t batch,
                                const void* d_q, void* d_out, float sm_scale, int32_t flags,
                                void* d_workspace, size_t workspace_bytes, void* stream);

/* Kept-set selection per (sequence, KV head) ("KV Cache optimization
 * techniques" 2.2 and 2.4; Technical Report 3.3 and 3.4).
 * Let S = pool slots, P = positions seen, ns = min(P, 4) sinks.
 *   H2O: if ns + S <= budget keep everything; otherwise keep the recent
 *     window (positions >= P - recent) and, of the other slots, the
 *     budget - 4 - recent with the highest score, ties to the lower position.
 *   StreamingLLM: if S <= window keep everything; otherwise keep positions
 *     >= P - window.
 * The sinks are always kept and are not part of the mask.
 *   d_keep_mask: u8 [batch][Hkv][max_blocks_per_seq*16], entry t = 1 if pool
 *   slot t is kept (entries >= S are left unspecified).
 * Records the plan (S, kept slots) that kvc_compact_blocks applies.
 * Errors: KVC_ERR_INVALID_ARG for a slice outside the cache, a null mask or
 * params, an unknown mode, a budget below 4 + recent, a negative recent
 * window, a StreamingLLM window below 1, a retention outside (0, 1], a bf16
 * window not covered by the recent window (H2O) or the StreamingLLM window,
 * or a short workspace;
 * KVC_ERR_UNSUPPORTED for block mode with a bf16 window or more than 4096
 * pages per sequence.  One launch (two in block mode). */
kvc_status kvc_h2o_select_evict(kvc_cache* cache, int32_t seq_begin, int32_t batch,
                                const kvc_evict_params* params, uint8_t* d_keep_mask,
                                void* d_workspace, size_t workspace_bytes, void* stream);

/* Block-granular eviction, KVC_EVICT_BLOCK (the eviction-and-reuse survey
 * page, section 4: blocks sorted by the mean attention score of their tokens,
 * the lowest int(n * (1 - ratio)) evicted).  A block is one page (16 slots)
 * of the sequence, shared by all KV heads.  The candidates are the n full
 * pages before the last `recent` pool slots; they are ordered by the sum, in
 * fp64 head by head and slot by slot, of their 16 x Hkv H2O scores (the sum
 * orders pages as the mean does), ties to the earlier page; the first
 * int(n * (1 - retention)) go.  kvc_h2o_select_evict writes the keep mask
 * (a page's slots all alike, every head alike) and the plan
 * S - 16 * evicted; kvc_compact_blocks then drops those pages from the
 * sequence's block-table row (the others keep their order), returns them to
 * the free stack and moves nothing in the pool.  The scores are what the
 * attention with KVC_ATTN_ACCUM_H2O accumulated.  At most 4096 pages per
 * sequence (max_blocks_per_seq), else KVC_ERR_UNSUPPORTED, before anything
 * is enqueued.  The selection takes two launches (the page sums over the
 * whole GPU, then one CTA per sequence selects and writes the mask; the page
 * sums use the workspace), the compaction one (the row rewrite). */

/* Compaction ("KV Cache optimization techniques" 2.2: gather the kept tokens;
 * 3.2: release blocks).  With S slots and n' < S kept, the kept slots are
 * gathered into the window [w, w + n'), w = 16 * floor((S - n') / 16), the
 * last page-aligned window of n' slots: every evicted slot inside the window
 * is filled, in ascending order, by the kept slots outside it, in ascending
 * order (codes, scales, position, score move together).  The block-table row
 * then drops its first w / 16 pages, so the window becomes slots [0, n'), and
 * the pages before and after the window return to the free stack.  After a
 * long context the always-kept recent tokens lie at the end, inside the
 * window, and do not move; at steady state (S = n' + 1) w = 0.  Attention is
 * invariant under the order of the attended tokens, so the result attends to
 * exactly the kept set.  Two launches (compaction, page release).
 *   d_keep_mask: the mask kvc_h2o_select_evict wrote for the same slice.
 * Errors: KVC_ERR_STATE if the slice has no pending selection. */
kvc_status kvc_compact_blocks(kvc_cache* cache, int32_t seq_begin, int32_t batch,
                              const uint8_t* d_keep_mask, void* d_workspace,
                              size_t workspace_bytes, void* stream);

/* Decode attention without a caller-supplied workspace.  The pages have no
 * counterpart to this call: it exists for callers that cannot allocate device
 * memory when they run a step (a fixed memory budget set at start-up, a
 * runtime that forbids allocation after initialisation, a host that owns
 * every allocation and passes plug-ins only their inputs and outputs).
 * Same arguments and results as kvc_decode_attention, which it calls; the
 * workspace is a fixed array of KVC_NOALLOC_SCRATCH_BYTES bytes inside the
 * library's device image, reserved on every GPU that loads the library and
 * held until the process exits.  It allocates nothing and calls no
 * allocating routine.
 *   - Returns KVC_ERR_CAPACITY, before anything is enqueued, when the slice
 *     needs more workspace than that (kvc_workspace_bytes(cache, batch) >
 *     KVC_NOALLOC_SCRATCH_BYTES); use kvc_decode_attention then.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it for the life of the process; make
 *     that first call before any stream capture on the device.  A device
 *     reset (cudaDeviceReset, or the primary context torn down and created
 *     again) unloads the library's module and invalidates the cached
 *     address: do not call this entry point on that device after one.
 *   - All calls share the one array and leave their contents in it; calls
 *     that overlap on the GPU (other streams or host threads) race.  No part
 *     of it needs to start at zero. */
#define KVC_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
kvc_status kvc_decode_attention_noalloc(kvc_cache* cache, int32_t seq_begin, int32_t batch,
                                        const void* d_q, void* d_out, float sm_scale, int32_t flags,
                                        void* stream);

/* One whole decode step of a layer in one call: append one token per
 * sequence (as kvc_quantize_append with n_new = 1), then decode attention
 * (H2O accumulation on in H2O and block mode, off in StreamingLLM mode),
 * selection and compaction with `params`, exactly as the four calls above
 * compute them.  After the split-K attention, the merge, the score update,
 * the selection and the compaction lists of each (sequence, KV head) run in
 * one kernel that keeps the scores, keys and keep decisions on chip; the row
 * moves follow in a launch of their own when some (sequence, KV head) moves
 * more than 32 rows (the first step after a long prompt), else that kernel
 * moves them itself (the steady state moves one row).  Three or four
 * launches in all (the split kernel runs even when every pool is empty: its
 * first CTA publishes the page prefix the next kernel reads); one more with
 * a bf16 window (its attention follows the split).  In block mode
 * (KVC_EVICT_BLOCK) that kernel stops after the scores; the page sums and
 * then the page selection and the row rewrite of each sequence follow (five
 * launches).  A CUDA graph captured at one state replays correctly at any
 * other (every kernel reads the lengths from the device; a post kernel
 * captured without a move kernel moves any number of rows itself).
 *   d_q: bf16 [batch][Hq][128]; d_k_new, d_v_new: bf16 [batch][Hkv][1][128];
 *   d_out: bf16 [batch][Hq][128]; workspace as for kvc_decode_attention.
 * Host-visible errors (arguments, capacity) are returned before anything is
 * enqueued.  No keep mask is written. */
kvc_status kvc_decode_step(kvc_cache* cache, int32_t seq_begin, int32_t batch, const void* d_q,
                           const void* d_k_new, const void* d_v_new, void* d_out, float sm_scale,
                           const kvc_evict_params* params, void* d_workspace, size_t workspace_bytes,
                           void* stream);

/* kvc_decode_step with the eviction off the output's path: the same results,
 * bit for bit.  On `stream`: the append, the split-K attention and the merge
 * (the outputs in d_out, each query head's softmax max and sum, and the sink
 * scores).  On `evict_stream`, after the merge (an event the library
 * records): the pool's (and the bf16 window's) score update, the selection,
 * the compaction lists and the row moves.  What the caller enqueues next on
 * `stream` (the next layer) overlaps the eviction.
 *   - The workspace stays in use until the eviction has run: give every
 *     cache (layer) its own.  d_q, d_k_new and d_v_new are read on `stream`
 *     only.
 *   - Every later call on this cache orders itself after the eviction: when
 *     both are eager, or both inside the same stream capture, through the
 *     library's event; an eviction enqueued eagerly is waited for from inside
 *     a capture as an external event node.  An eviction captured into a
 *     graph is ordered by the graph: before its capture ends, the caller
 *     joins `evict_stream` back into the capturing stream (an event recorded
 *     on `evict_stream` and waited on by `stream`), as CUDA requires.
 *   - kvc_read_status, kvc_cache_sync_host and kvc_cache_reset on this cache
 *     wait for the eviction on their stream.
 *   - evict_stream may equal stream (then nothing overlaps).
 * Launches: the four or five of kvc_decode_step, plus the merge. */
kvc_status kvc_decode_step_overlap(kvc_cache* cache, int32_t seq_begin, int32_t batch, const void* d_q,
                                   const void* d_k_new, const void* d_v_new, void* d_out, float sm_scale,
                                   const kvc_evict_params* params, void* d_workspace, size_t workspace_bytes,
                                   void* stream, void* evict_stream);

/* Prefill of fresh sequences (the step before the decode path): append the
 * n prompt tokens of every sequence of the slice (exactly as
 * kvc_quantize_append), run the causal attention of the n queries over the
 * prompt's exact bf16 keys and values (query i attends keys 0..i; query head
 * j reads KV head j / G), and, with KVC_ATTN_ACCUM_H2O, set every prompt
 * token's H2O score (sinks, pool slots, bf16 window) to the sum over all n
 * queries and the G query heads of its KV head of the probability they give
 * it: the column sums of the prompt's attention matrix (Technical Report 3.4:
 * scores = attention_scores.sum(dim=0); the eviction-and-reuse survey page
 * 3.3: a token's cumulative attention from the later tokens).
 *   d_q:   bf16 [batch][Hq][n][128];  d_k, d_v: bf16 [batch][Hkv][n][128];
 *   d_out: bf16 [batch][Hq][n][128];  all 16-byte aligned;
 *   d_workspace: kvc_prefill_workspace_bytes(cache, batch, n) bytes, 256-byte
 *   aligned (the row statistics the score pass reads).
 * Two or three launches (append, attention, scores), tensor cores (bf16
 * operands, fp32 accumulation).  Errors: KVC_ERR_STATE unless every sequence
 * of the slice is empty (no token appended since the last reset);
 * KVC_ERR_CAPACITY as kvc_quantize_append. */
size_t kvc_prefill_workspace_bytes(const kvc_cache* cache, int32_t batch, int32_t n);
kvc_status kvc_prefill_attention(kvc_cache* cache, int32_t seq_begin, int32_t batch, int32_t n, const void* d_q,
                                 const void* d_k, const void* d_v, void* d_out, float sm_scale, int32_t flags,
                                 void* d_workspace, size_t workspace_bytes, void* stream);

/* A prompt of n tokens appended to sequences that may already hold context
 * (a later turn), attending to the compressed cache: append the tokens (as
 * kvc_quantize_append), then prompt query i (position P + i, P the positions
 * seen before) attends, as a decode step does, to every held token at a
 * position <= P + i in its stored form (sinks bf16, pool tokens dequantised),
 * and with KVC_ATTN_ACCUM_H2O adds its probabilities to their H2O scores (the
 * survey's prefill over the compressed pool: "KV cache eviction and reuse
 * survey" 3.3, cumulative attention from the later tokens; Technical Report
 * 3.4, column sums of the attention matrix).  Because the prompt's own pool
 * tokens are the last pool slots, what query i sees is the sinks up to its
 * position and a prefix of the pool: the causal mask shifted by the context.
 * Three launches: the append, then a multi-query kernel in two passes (the
 * row maxima and sums; the outputs and per-CTA column sums, the last CTA of
 * each (sequence, KV head) adding them, in a fixed order, to the scores).
 * Every pool page is read once per pass per tile of 64 attention rows (query
 * x query head of the group); tensor cores, the codes entering the MMA as in
 * kvc_decode_attention.
 *   d_q:   bf16 [batch][Hq][n][128];  d_k, d_v: bf16 [batch][Hkv][n][128];
 *   d_out: bf16 [batch][Hq][n][128];  all device memory, 16-byte aligned,
 *   owned by the caller; flags 0 or KVC_ATTN_ACCUM_H2O; d_workspace:
 *   kvc_prefill_context_workspace_bytes(cache, batch, n) bytes, 256-byte
 *   aligned (scratch for the duration of the call, stream-ordered: per
 *   (sequence, KV head) the n * G row statistics and up to 64 rows of
 *   column sums over 4 + max_blocks_per_seq * 16 tokens).
 * Errors, before any launch: KVC_ERR_INVALID_ARG (range, n <= 0, flags,
 * sm_scale not positive and finite, pointers, workspace);
 * KVC_ERR_CAPACITY as kvc_quantize_append; KVC_ERR_UNSUPPORTED with a bf16
 * window (bf16_window > 0) or n * Hq > 2^30.  KVC_ERR_CUDA when a launch
 * fails; the lengths then already include the appended prompt. */
size_t kvc_prefill_context_workspace_bytes(const kvc_cache* cache, int32_t batch, int32_t n);
kvc_status kvc_prefill_context(kvc_cache* cache, int32_t seq_begin, int32_t batch, int32_t n, const void* d_q,
                               const void* d_k, const void* d_v, void* d_out, float sm_scale, int32_t flags,
                               void* d_workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- misc ---- */

/* Synchronise `stream`, copy the device status word to *h_status and clear
 * it.  Returns KVC_ERR_DEVICE when any bit was set. */
kvc_status kvc_read_status(kvc_cache* cache, int32_t* h_status, void* stream);

/* Tracing: when both are non-NULL, the next kvc_decode_attention calls record
 * `ev_start` (a cudaEvent_t) just before the split-K attention kernel and
 * `ev_stop` just after it, on the call's stream (kvc_decode_step and
 * kvc_prefill_context likewise, around each split launch;
 * kvc_prefill_attention around its attention kernel, outside any stream
 * capture).  NULL, NULL turns it off. */
kvc_status kvc_set_trace_events(kvc_cache* cache, void* ev_start, void* ev_stop);

/* Number of kernels the last call on this handle enqueued. */
int32_t kvc_last_launch_count(const kvc_cache* cache);

const char* kvc_status_string(kvc_status status);

/* Library version: major * 10000 + minor * 100 + patch.  A caller built
 * against this header checks kvc_version() == KVC_VERSION before passing
 * structures (kvc_config grew in 0.2: bf16_window, codes;
 * kvc_prefill_context_workspace_bytes took the prompt length in 0.3;
 * 0.4 added kvc_decode_step_overlap). */
#define KVC_VERSION 400
int32_t kvc_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KVC_H */
