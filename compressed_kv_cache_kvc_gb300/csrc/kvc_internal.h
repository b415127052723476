// Internal declarations shared by the host side (kvc_host.cpp) and the
// kernels (kvc_*.cu) of the compressed-KV library.  Not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kvc {

constexpr int kHeadDim = 128;
constexpr int kPage = 16;
constexpr int kSinks = 4;
constexpr int kMaxGroup = 8;     // query heads per KV head handled by one MMA column tile
constexpr int kCounters = 64;    // int32 counters block

// Device view of one layer's cache state (passed to kernels by value).
struct DevState {
  uint8_t* k_codes;     // [num_blocks][hkv][16][row_bytes]
  uint8_t* v_codes;
  float* k_scale;       // [num_blocks][hkv][16]
  float* v_scale;
  int32_t* slot_pos;
  float* score;
  uint16_t* sink_k;     // [max_batch][hkv][4][128] bf16
  uint16_t* sink_v;
  float* sink_score;    // [max_batch][hkv][4]
  int32_t* block_table; // [max_batch][max_bps]
  int32_t* seq_slots;   // [max_batch]
  int32_t* seq_pos;     // [max_batch]
  int32_t* free_stack;  // [num_blocks]
  int32_t* counters;    // [0] free top, [1] status
  int32_t* plan;        // [max_batch][2]
  uint16_t* ring_k;     // [max_batch][hkv][ring][128] bf16 (hybrid precision window)
  uint16_t* ring_v;
  float* ring_score;    // [max_batch][hkv][ring]
  int32_t hq, hkv, group, bits, row_bytes, num_blocks, max_batch, max_bps;
  int32_t ring;         // hybrid window W (0: off); ring slot of position p >= 4 is (p - 4) % W
  int32_t fp8;          // 1: FP8 E4M3 codes (bits = 8), 0: integer codes
};

// Tokens held in the bf16 window of a sequence with P positions.
__host__ __device__ inline int ring_count(int P, int W) {
  if (W <= 0 || P <= kSinks) return 0;
  return P - kSinks < W ? P - kSinks : W;
}

// Positions [pool_lo, pool_hi) enter the pool when n_new tokens are appended
// to a sequence that has seen P: with a window, the tokens that leave it
// (from the ring, then straight from the input), else every non-sink token.
__host__ __device__ inline void pool_range(int P, int n_new, int W, int* lo, int* hi) {
  const int a = P - W > kSinks ? P - W : kSinks;
  const int e = P + n_new - W;
  *lo = a;
  *hi = e > a ? e : a;
}

enum { kCtrFreeTop = 0, kCtrStatus = 1 };

// Status bits (mirror kvc.h).
constexpr int kDevOutOfBlocks = 0x1;
constexpr int kDevBadBlockId = 0x2;
constexpr int kDevBadKeepMask = 0x4;
constexpr int kDevTableOverflow = 0x8;
constexpr int kDevStackOverflow = 0x10;
constexpr int kDevStaleHost = 0x20;
constexpr int kDevWaitTimeout = 0x40;
constexpr int kDevPrefillRange = 0x80;

// Scratch carved from the caller's workspace for one attention call.
//
// Work split ("stream-K"): the pages of all (sequence, KV head) pairs of the
// slice are laid end to end (pair p = local_seq * hkv + head, pages in order)
// and CTA i of the N-CTA grid takes pages [floor(i*T/N), floor((i+1)*T/N)).
// A CTA writes one partial (m, l, o) per pair it touches, into partial slot
// p + i; the slots of different (pair, CTA) combinations never collide
// because both orders run along the same page sequence.
struct AttnWork {
  float* part_o;    // [pairs + ncta][group][128]
  float* part_ml;   // [pairs + ncta][group][2]
  float* logits;    // [batch][hkv][group][s_cap]  (log2 domain)
  float* stats;     // [batch][hq][2]  global (M, L) per query head
  int* cum;         // [batch + 1] page prefix of the slice (written by split CTA 0)
  int* seq_ticket;  // [batch] per-sequence completion tickets (zeroed by split CTA 0)
  float* ring_po;   // [batch][hkv][ring_chunks][group][128] partials of the bf16 window
  float* ring_pml;  // [batch][hkv][ring_chunks][group][2]
  float* ring_lg;   // [batch][hkv][group][ring] window logits (log2 domain)
  int ring_chunks;  // ceil(W / kRingChunk), 0 without a window
  int ncta;         // grid size of the split kernel
  int s_cap;
};

constexpr int kMaxCallBatch = 1024;  // sequences per attention call (prefix table in shared memory)
constexpr int kRingChunk = 64;       // window slots per CTA of the window attention
constexpr int kMaxRing = 4096;
constexpr int kMaxSplitCtas = 2048;

// Raise a kernel's dynamic shared-memory limit to `bytes`, once per device
// (`done` holds one flag per device ordinal below 64).  Needed whenever the
// kernel's static plus dynamic shared memory passes the 48 KB default.
inline cudaError_t opt_in_smem(const void* fn, int bytes, int* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev < 64) done[dev] = 1;
  return e;
}

// ---- launchers (return cudaGetLastError of the launch) -------------------
cudaError_t launch_append(const DevState& s, int seq_begin, int batch, int n_new,
                          const uint16_t* k, const uint16_t* v, cudaStream_t st);
// Two launches (page allocation, then the rows over token chunks) for long
// appends that push no bf16-window token into the pool.
cudaError_t launch_append_bulk(const DevState& s, int seq_begin, int batch, int n_new, const uint16_t* k,
                               const uint16_t* v, cudaStream_t st);
constexpr int kBulkAppendMin = 64;  // tokens per sequence from which the bulk path pays
cudaError_t launch_fill_free_stack(const DevState& s, cudaStream_t st);

cudaError_t launch_attention_split(const DevState& s, int seq_begin, int batch, const uint16_t* q,
                                   float qk_scale_log2, const AttnWork& w, bool spill_logits,
                                   cudaStream_t st);
// Attention over the bf16 window (hybrid precision): one partial per
// (sequence, KV head, chunk of kRingChunk slots), logits to w.ring_lg.
cudaError_t launch_attention_ring(const DevState& s, int seq_begin, int batch, const uint16_t* q,
                                  float qk_scale_log2, const AttnWork& w, cudaStream_t st);
// scores: which H2O scores the merge adds (the sink scores need the query).
enum MergeScores { kMergeNoScores = 0, kMergeAllScores = 1, kMergeSinkScores = 2 };
cudaError_t launch_attention_merge(const DevState& s, int seq_begin, int batch, const uint16_t* q,
                                   uint16_t* out, float qk_scale_log2, const AttnWork& w, MergeScores scores,
                                   cudaStream_t st);

struct SelectArgs {
  int mode, budget, recent, window;
  int s_cap;            // mask row stride
  int smem_slots;       // > 0: keys/pos staged in shared memory (capacity in slots)
  uint32_t* g_keys;     // global fallback [batch][hkv][s_cap]
  int32_t* g_pos;
};
cudaError_t launch_select(const DevState& s, int seq_begin, int batch, const SelectArgs& a,
                          uint8_t* keep_mask, cudaStream_t st);

// Block-granular eviction.  keys: [batch][max_bps] page keys in the
// workspace (block_keys writes them); select writes the plan and the keep
// mask, release applies a keep mask, evict selects and applies in one launch.
// At most kMaxBlockPages pages per sequence.
constexpr int kMaxBlockPages = 4096;
cudaError_t launch_block_keys(const DevState& s, int seq_begin, int batch, int recent, int max_cand,
                              unsigned long long* keys, cudaStream_t st);
cudaError_t launch_select_blocks(const DevState& s, int seq_begin, int batch, int recent, double retention,
                                 const unsigned long long* keys, uint8_t* keep_mask, int s_cap, cudaStream_t st);
cudaError_t launch_evict_blocks(const DevState& s, int seq_begin, int batch, int recent, double retention,
                                const unsigned long long* keys, cudaStream_t st);
cudaError_t launch_release_blocks(const DevState& s, int seq_begin, int batch, const uint8_t* keep_mask,
                                  int s_cap, cudaStream_t st);
// Whole sequences back to the pool (kvc_release_sequences).
cudaError_t launch_release_sequences(const DevState& s, int seq_begin, int batch, cudaStream_t st);
// g_holes / g_srcs: [batch][hkv][s_cap] move lists in the workspace, used when
// smem_moves == 0; otherwise both lists (smem_moves entries each) live in
// shared memory.
cudaError_t launch_compact(const DevState& s, int seq_begin, int batch, const uint8_t* keep_mask,
                           int s_cap, int32_t* g_holes, int32_t* g_srcs, int smem_moves, cudaStream_t st);
int compact_max_smem_moves();

// Prefill of fresh sequences: causal attention over the prompt's bf16 K/V
// (output bf16 [batch][hq][n][128], row statistics to `stats`
// [batch][hq][n][2]) and, with `scores`, the H2O scores of its tokens.
// The forward on tcgen05 (kvc_prefill_tc.cu): outputs and row statistics as
// the mma.sync forward's.
cudaError_t launch_prefill_fwd_tc(const DevState& s, int batch, int n, const uint16_t* q, const uint16_t* k,
                                  const uint16_t* v, uint16_t* out, float* stats, float qk_scale_log2,
                                  cudaStream_t st);
int prefill_fwd_tc_smem_bytes();
cudaError_t launch_prefill_scores_tc(const DevState& s, int seq_begin, int batch, int n, const uint16_t* q,
                                    const uint16_t* k, const float* stats, float qk_scale_log2, cudaStream_t st);
cudaError_t launch_prefill(const DevState& s, int seq_begin, int batch, int n, const uint16_t* q, const uint16_t* k,
                           const uint16_t* v, uint16_t* out, float* stats, float qk_scale_log2, bool scores,
                           cudaStream_t st, cudaEvent_t trace_start = nullptr,
                           cudaEvent_t trace_stop = nullptr);

// A prompt on sequences with context (kvc_prefill_context), after its
// append: the multi-query attention over the compressed cache in two
// launches (row statistics; outputs, column sums and, with `accumulate`, the
// scores).  stats: [batch * hkv][n * group][2] floats; colsum: [batch * hkv]
// [ctx_groups][4 + s_cap] floats; ticket: [batch * hkv] ints.
constexpr int kCtxBtStage = 2048;   // block-table entries staged in shared memory
constexpr int kMaxCtxGroups = 64;   // CTAs per (sequence, KV head)
int ctx_groups(int n, int group);
cudaError_t launch_ctx_attention(const DevState& s, int seq_begin, int batch, int n, const uint16_t* q,
                                 uint16_t* out, float* stats, float* colsum, int* ticket, int s_cap,
                                 float qk_scale_log2, bool accumulate, cudaStream_t st);

// Fused merge + H2O scores + selection + compaction (kvc_decode_step).
struct StepArgs {
  int mode, budget, recent, window;
  int s_cap;            // row stride of the workspace key/position arrays
  int smem_slots;       // > 0: keys (and, with pos_smem, positions) in shared memory (capacity in slots)
  int pos_smem;         // positions in shared memory too (else in g_pos)
  uint32_t* g_keys;     // global fallback [batch][hkv][s_cap]; then the hole list
  int32_t* g_pos;       // likewise; then the source list
  int* n_moves;         // [batch][hkv] list lengths (post kernel -> move kernel)
  int inline_moves;     // the post kernel moves the rows itself (no move kernel follows)
  int merged;           // the merge (and the sink scores) already ran: read each head's (M, L) from w.stats
};
// Pairs that move at most this many rows are moved inside the post kernel
// (the steady state moves one row per pair).
constexpr int kInlineMoves = 32;
cudaError_t launch_step_post(const DevState& s, int seq_begin, int batch, const uint16_t* q, uint16_t* out,
                             float qk_scale_log2, const AttnWork& w, const StepArgs& a, int sm_count,
                             cudaStream_t st);
// max_moves: an upper bound of any pair's move count (sizes the grid only)
cudaError_t launch_step_moves(const DevState& s, int batch, const StepArgs& a, int sm_count, int max_moves,
                              cudaStream_t st);
int step_max_smem_bytes();  // dynamic shared memory of the post kernel (a multiple of 16)

int attention_smem_bytes(int bits);
int attention_ctas_per_sm(int bits, bool fp8);  // resident split CTAs per SM (occupancy API, cached)
int select_max_smem_slots();

}  // namespace kvc
