// Host side of the C ABI (include/kvc.h): argument validation, the host mirror
// of the sequence lengths (so that capacity errors are caught before anything
// is enqueued, as the paged cache's allocate_sequence returns False in
// "KV Cache optimization techniques" section 3.2), buffer carving, the split-K
// launch policy, and the kernel launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/kvc.h"
#include "kvc_internal.h"

using kvc::DevState;

namespace {

constexpr size_t kAlign = 256;
// A split CTA has fixed costs (the page prefix, the query fragments, the
// ring's first copies, the CTA merge and its partial): small steps (the
// steady state of a long context, ~6500 pages) run faster on fewer, fuller
// CTAs (at least 32 pages each: 58.0 ms for the 32k-context stack's 64 steps,
// against 66.5 ms with 4, 65.2 with 16 and 59.3 with 64), down to one CTA
// per SM; large steps fill one wave either way.
constexpr int kMinPagesPerCta = 32;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Layout {
  size_t off[KVC_BUF_COUNT];
  size_t size[KVC_BUF_COUNT];
  size_t total;
};

bool config_valid(const kvc_config* c) {
  return c && c->num_q_heads > 0 && c->num_kv_heads > 0 && c->num_blocks > 0 && c->max_batch > 0 &&
         c->max_blocks_per_seq > 0 && c->num_q_heads % c->num_kv_heads == 0;
}

kvc_status config_check(const kvc_config* c) {
  if (!config_valid(c)) return KVC_ERR_INVALID_ARG;
  if (c->head_dim != kvc::kHeadDim || c->page_size != kvc::kPage || (c->bits != 8 && c->bits != 4) ||
      c->num_q_heads / c->num_kv_heads > kvc::kMaxGroup)
    return KVC_ERR_UNSUPPORTED;
  if (c->bf16_window < 0) return KVC_ERR_INVALID_ARG;
  if (c->codes != KVC_CODES_INT && c->codes != KVC_CODES_E4M3) return KVC_ERR_INVALID_ARG;
  if (c->codes == KVC_CODES_E4M3 && c->bits != 8) return KVC_ERR_UNSUPPORTED;
  if (c->bf16_window > kvc::kMaxRing) return KVC_ERR_UNSUPPORTED;
  // 32-bit slot arithmetic inside the kernels
  if ((double)c->num_blocks * c->num_kv_heads * kvc::kPage >= 2147483647.0 ||
      (double)c->max_blocks_per_seq * kvc::kPage > 2.0e9)
    return KVC_ERR_UNSUPPORTED;
  return KVC_OK;
}

Layout make_layout(const kvc_config* c) {
  Layout L{};
  const size_t slots = (size_t)c->num_blocks * c->num_kv_heads * kvc::kPage;
  const size_t row_bytes = (size_t)kvc::kHeadDim * c->bits / 8;
  const size_t sinks = (size_t)c->max_batch * c->num_kv_heads * kvc::kSinks;
  L.size[KVC_BUF_K_CODES] = slots * row_bytes;
  L.size[KVC_BUF_V_CODES] = slots * row_bytes;
  L.size[KVC_BUF_K_SCALE] = slots * 4;
  L.size[KVC_BUF_V_SCALE] = slots * 4;
  L.size[KVC_BUF_SLOT_POS] = slots * 4;
  L.size[KVC_BUF_SCORE] = slots * 4;
  L.size[KVC_BUF_SINK_K] = sinks * kvc::kHeadDim * 2;
  L.size[KVC_BUF_SINK_V] = sinks * kvc::kHeadDim * 2;
  L.size[KVC_BUF_SINK_SCORE] = sinks * 4;
  L.size[KVC_BUF_BLOCK_TABLE] = (size_t)c->max_batch * c->max_blocks_per_seq * 4;
  L.size[KVC_BUF_SEQ_SLOTS] = (size_t)c->max_batch * 4;
  L.size[KVC_BUF_SEQ_POS] = (size_t)c->max_batch * 4;
  L.size[KVC_BUF_FREE_STACK] = (size_t)c->num_blocks * 4;
  L.size[KVC_BUF_COUNTERS] = (size_t)kvc::kCounters * 4;
  L.size[KVC_BUF_PLAN] = (size_t)c->max_batch * 2 * 4;
  const size_t ring = (size_t)c->max_batch * c->num_kv_heads * c->bf16_window;
  L.size[KVC_BUF_RING_K] = ring * kvc::kHeadDim * 2;
  L.size[KVC_BUF_RING_V] = ring * kvc::kHeadDim * 2;
  L.size[KVC_BUF_RING_SCORE] = ring * 4;
  size_t o = 0;
  for (int i = 0; i < KVC_BUF_COUNT; ++i) {
    L.off[i] = o;
    o = align_up(o + L.size[i]);
  }
  L.total = o;
  return L;
}

int pages_of(int slots) { return (slots + kvc::kPage - 1) / kvc::kPage; }

}  // namespace

struct kvc_cache {
  kvc_config cfg;
  Layout layout;
  uint8_t* base;
  DevState dev;
  std::vector<int32_t> slots;  // host mirror: pool slots per sequence
  std::vector<int32_t> pos;    // host mirror: positions seen per sequence
  // pending selection (kvc_h2o_select_evict -> kvc_compact_blocks)
  bool plan_pending = false;
  bool plan_block = false;  // the pending plan drops whole pages
  int32_t plan_begin = 0, plan_batch = 0;
  std::vector<int32_t> plan_new;
  void* trace_start = nullptr;
  void* trace_stop = nullptr;
  int32_t last_launches = 0;
  int sm_count = 0;
  // kvc_decode_step_overlap: the merge's completion (the eviction stream
  // waits for it) and the eviction's completion, still pending until a later
  // call on this cache orders itself after it (created at the first such call)
  cudaEvent_t merge_done = nullptr;
  cudaEvent_t evict_done = nullptr;
  bool evict_pending = false;
  bool evict_in_capture = false;      // recorded while the streams were being captured
  unsigned long long evict_capture_id = 0;
};

namespace {

int used_pages(const kvc_cache* c) {
  long long u = 0;
  for (int b = 0; b < c->cfg.max_batch; ++b) u += pages_of(c->slots[b]);
  return (int)u;
}

bool range_ok(const kvc_cache* c, int32_t seq_begin, int32_t batch) {
  return seq_begin >= 0 && batch > 0 && (long long)seq_begin + batch <= c->cfg.max_batch;
}

int s_cap(const kvc_cache* c) { return c->cfg.max_blocks_per_seq * kvc::kPage; }

// Workspace carving (all regions 256-byte aligned).
struct WsLayout {
  size_t part_o, part_ml, logits, stats, cum, ticket, moves, keys, pos, ring_po, ring_pml, ring_lg, total;
};

int ring_chunks(const kvc_cache* c);

WsLayout ws_layout(const kvc_cache* c, int batch) {
  const size_t G = c->cfg.num_q_heads / c->cfg.num_kv_heads;
  const size_t pairs = (size_t)batch * c->cfg.num_kv_heads;
  const size_t nslots = pairs + kvc::kMaxSplitCtas;  // stream-K partial slots
  const size_t cap = s_cap(c);
  WsLayout w{};
  size_t o = 0;
  w.part_o = o;
  o = align_up(o + nslots * G * kvc::kHeadDim * 4);
  w.part_ml = o;
  o = align_up(o + nslots * G * 2 * 4);
  w.logits = o;
  o = align_up(o + pairs * cap * G * 4);
  w.stats = o;
  o = align_up(o + (size_t)batch * c->cfg.num_q_heads * 2 * 4);
  w.cum = o;
  o = align_up(o + ((size_t)batch + 1) * 4);
  w.ticket = o;
  o = align_up(o + (size_t)batch * 4);
  w.moves = o;
  o = align_up(o + pairs * 4);
  w.keys = o;
  o = align_up(o + pairs * cap * 4);
  w.pos = o;
  o = align_up(o + pairs * cap * 4);
  const size_t rc = ring_chunks(c);
  w.ring_po = o;
  o = align_up(o + pairs * rc * G * kvc::kHeadDim * 4);
  w.ring_pml = o;
  o = align_up(o + pairs * rc * G * 2 * 4);
  w.ring_lg = o;
  o = align_up(o + pairs * G * (size_t)c->cfg.bf16_window * 4);
  w.total = o;
  return w;
}

int ring_chunks(const kvc_cache* c) {
  return (c->cfg.bf16_window + kvc::kRingChunk - 1) / kvc::kRingChunk;
}

int sm_count(kvc_cache* c) {
  if (c->sm_count <= 0) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
      c->sm_count = n;
    else
      c->sm_count = 152;
  }
  return c->sm_count;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Checks shared by kvc_decode_attention and kvc_decode_step (everything the
// host can see before a launch).  `appended` tokens are about to be added to
// every sequence of the slice before the attention runs.
kvc_status attention_check(const kvc_cache* c, int32_t seq_begin, int32_t batch, const void* d_q, const void* d_out,
                           float sm_scale, const void* d_workspace, size_t workspace_bytes, int appended) {
  if (!range_ok(c, seq_begin, batch)) return KVC_ERR_INVALID_ARG;
  if (!d_q || !d_out || !aligned(d_q, 16) || !aligned(d_out, 16)) return KVC_ERR_INVALID_ARG;
  if (!(sm_scale > 0.0f) || !std::isfinite(sm_scale)) return KVC_ERR_INVALID_ARG;
  const WsLayout wl = ws_layout(c, batch);
  if (!d_workspace || !aligned(d_workspace, kAlign) || workspace_bytes < wl.total) return KVC_ERR_INVALID_ARG;
  if (batch > kvc::kMaxCallBatch) return KVC_ERR_UNSUPPORTED;
  for (int i = 0; i < batch; ++i)
    if (c->pos[seq_begin + i] + appended <= 0) return KVC_ERR_INVALID_ARG;  // nothing to attend to
  return KVC_OK;
}

// Stream-K grid and workspace carving of one attention call (host mirror
// lengths as they are now).
void attention_plan(kvc_cache* c, int32_t seq_begin, int32_t batch, void* d_workspace, kvc::AttnWork* w,
                    long long* total_pages) {
  const WsLayout wl = ws_layout(c, batch);
  long long tp = 0;
  for (int i = 0; i < batch; ++i) tp += (long long)pages_of(c->slots[seq_begin + i]) * c->cfg.num_kv_heads;
  // one wave of resident CTAs, each with at least kMinPagesPerCta pages of the
  // current lengths (any grid size is correct for any lengths, so a graph
  // replayed at other lengths stays correct)
  int ncta = 1;
  if (tp > 0) {
    ncta = sm_count(c) * kvc::attention_ctas_per_sm(c->cfg.bits, c->cfg.codes == KVC_CODES_E4M3);
    // fuller CTAs, but no fewer than one per SM while each still gets 4 pages
    const long long want = std::max<long long>(tp / kMinPagesPerCta, std::min<long long>(sm_count(c), tp / 4));
    ncta = (int)std::min<long long>(ncta, std::max<long long>(1, want));
    ncta = std::max(1, std::min(ncta, kvc::kMaxSplitCtas));
  }
  uint8_t* ws = static_cast<uint8_t*>(d_workspace);
  *w = kvc::AttnWork{};
  w->part_o = reinterpret_cast<float*>(ws + wl.part_o);
  w->part_ml = reinterpret_cast<float*>(ws + wl.part_ml);
  w->logits = reinterpret_cast<float*>(ws + wl.logits);
  w->stats = reinterpret_cast<float*>(ws + wl.stats);
  w->cum = reinterpret_cast<int*>(ws + wl.cum);
  w->seq_ticket = reinterpret_cast<int*>(ws + wl.ticket);
  w->ring_po = reinterpret_cast<float*>(ws + wl.ring_po);
  w->ring_pml = reinterpret_cast<float*>(ws + wl.ring_pml);
  w->ring_lg = reinterpret_cast<float*>(ws + wl.ring_lg);
  w->ring_chunks = ring_chunks(c);
  w->ncta = ncta;
  w->s_cap = s_cap(c);
  *total_pages = tp;
}

// The split-K attention launch, bracketed by the trace events when set (under
// stream capture they become event-record nodes of the graph).
// With no pages the launch is skipped unless `always` (kvc_decode_step: the
// post kernel reads the page prefix and tickets that the split's first CTA
// publishes, and a grid of one CTA with no pages does only that).
kvc_status launch_split_traced(kvc_cache* c, int32_t seq_begin, int32_t batch, const void* d_q, float qk_scale_log2,
                               const kvc::AttnWork& w, bool h2o, long long total_pages, cudaStream_t st,
                               int* launches, bool always = false) {
  if (total_pages <= 0 && !always) return KVC_OK;
  const bool trace = c->trace_start && c->trace_stop;
  unsigned rec_flags = cudaEventRecordDefault;
  if (trace) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return KVC_ERR_CUDA;
    if (cs == cudaStreamCaptureStatusActive) rec_flags = cudaEventRecordExternal;
  }
  if (trace && cudaEventRecordWithFlags(static_cast<cudaEvent_t>(c->trace_start), st, rec_flags) != cudaSuccess)
    return KVC_ERR_CUDA;
  if (kvc::launch_attention_split(c->dev, seq_begin, batch, static_cast<const uint16_t*>(d_q), qk_scale_log2, w, h2o,
                                  st) != cudaSuccess)
    return KVC_ERR_CUDA;
  ++*launches;
  if (trace && cudaEventRecordWithFlags(static_cast<cudaEvent_t>(c->trace_stop), st, rec_flags) != cudaSuccess)
    return KVC_ERR_CUDA;
  return KVC_OK;
}

// The attention over the bf16 window (hybrid precision), when there is one.
kvc_status launch_ring(kvc_cache* c, int32_t seq_begin, int32_t batch, const void* d_q, float qk_scale_log2,
                       const kvc::AttnWork& w, cudaStream_t st, int* launches) {
  if (c->cfg.bf16_window <= 0) return KVC_OK;
  if (kvc::launch_attention_ring(c->dev, seq_begin, batch, static_cast<const uint16_t*>(d_q), qk_scale_log2, w,
                                 st) != cudaSuccess)
    return KVC_ERR_CUDA;
  ++*launches;
  return KVC_OK;
}

// Kept slots per sequence after a selection (the host mirror's plan).
// The window W of hybrid precision is always kept: the recent window (H2O)
// or the StreamingLLM window must cover it.
kvc_status evict_check(const kvc_cache* c, const kvc_evict_params* p) {
  if (!p) return KVC_ERR_INVALID_ARG;
  const int W = c->cfg.bf16_window;
  if (p->mode == KVC_EVICT_H2O) {
    if (p->recent < W || p->budget < kvc::kSinks + p->recent) return KVC_ERR_INVALID_ARG;
  } else if (p->mode == KVC_EVICT_STREAMING) {
    if (p->window < 1 || p->window < W) return KVC_ERR_INVALID_ARG;
  } else if (p->mode == KVC_EVICT_BLOCK) {
    if (p->recent < 0 || !(p->retention > 0.0 && p->retention <= 1.0)) return KVC_ERR_INVALID_ARG;
    if (W > 0) return KVC_ERR_UNSUPPORTED;
  } else {
    return KVC_ERR_INVALID_ARG;
  }
  return KVC_OK;
}

// Candidate pages of block-granular eviction, the most of any sequence of
// the slice (sizes the page-key grid only).
int max_block_cand(const kvc_cache* c, int32_t seq_begin, int32_t batch, int recent) {
  int m = 0;
  for (int i = 0; i < batch; ++i) m = std::max(m, std::max(0, c->slots[seq_begin + i] - recent) / kvc::kPage);
  return m;
}

// Pool slots kept out of S; the nr window tokens count inside the budget or
// window.
int plan_keep(const kvc_evict_params* p, int S, int P, int W) {
  const int ns = std::min(P, kvc::kSinks);
  const int nr = kvc::ring_count(P, W);
  if (p->mode == KVC_EVICT_H2O) return (ns + nr + S <= p->budget) ? S : p->budget - kvc::kSinks - nr;
  if (p->mode == KVC_EVICT_BLOCK) {
    // the device computes the same double expression
    const int n_cand = std::max(0, S - p->recent) / kvc::kPage;
    const int n_evict = (int)((double)n_cand * (1.0 - p->retention));
    return S - kvc::kPage * n_evict;
  }
  return (nr + S <= p->window) ? S : p->window - nr;
}

}  // namespace

extern "C" {

namespace {

// Every call that touches a cache first orders `st` after the eviction a
// kvc_decode_step_overlap call left running on its eviction stream: eager
// after eager, or within one stream capture (a graph edge).  An eviction
// recorded eagerly is waited for from inside a capture as an external event
// node.  An eviction recorded in a capture belongs to that graph: its
// launches are ordered by the caller, and the graph joins its eviction
// stream before the capture ends.
kvc_status order_after_eviction(kvc_cache* c, cudaStream_t st) {
  if (!c->evict_pending) return KVC_OK;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  unsigned long long id = 0;
  if (cudaStreamGetCaptureInfo(st, &cs, &id) != cudaSuccess) return KVC_ERR_CUDA;
  const bool cap = cs == cudaStreamCaptureStatusActive;
  cudaError_t e = cudaSuccess;
  if (!cap && !c->evict_in_capture)
    e = cudaStreamWaitEvent(st, c->evict_done, 0);
  else if (cap && !c->evict_in_capture)
    e = cudaStreamWaitEvent(st, c->evict_done, cudaEventWaitExternal);
  else if (cap && id == c->evict_capture_id)
    e = cudaStreamWaitEvent(st, c->evict_done, 0);
  return e == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

}  // namespace

int32_t kvc_version(void) { return KVC_VERSION; }

const char* kvc_status_string(kvc_status s) {
  switch (s) {
    case KVC_OK: return "ok";
    case KVC_ERR_INVALID_ARG: return "invalid argument";
    case KVC_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVC_ERR_CAPACITY: return "out of cache capacity";
    case KVC_ERR_CUDA: return "CUDA runtime error";
    case KVC_ERR_DEVICE: return "device reported an error";
    case KVC_ERR_STATE: return "call order violated";
  }
  return "unknown status";
}

size_t kvc_state_bytes(const kvc_config* cfg) {
  if (config_check(cfg) != KVC_OK) return 0;
  return make_layout(cfg).total;
}

kvc_status kvc_cache_create(const kvc_config* cfg, void* d_state, size_t state_bytes, kvc_cache** out) {
  if (!out) return KVC_ERR_INVALID_ARG;
  *out = nullptr;
  const kvc_status st = config_check(cfg);
  if (st != KVC_OK) return st;
  const Layout L = make_layout(cfg);
  if (!d_state || !aligned(d_state, kAlign) || state_bytes < L.total) return KVC_ERR_INVALID_ARG;
  kvc_cache* c = new (std::nothrow) kvc_cache();
  if (!c) return KVC_ERR_INVALID_ARG;
  c->cfg = *cfg;
  c->layout = L;
  c->base = static_cast<uint8_t*>(d_state);
  DevState& d = c->dev;
  uint8_t* b = c->base;
  d.k_codes = b + L.off[KVC_BUF_K_CODES];
  d.v_codes = b + L.off[KVC_BUF_V_CODES];
  d.k_scale = reinterpret_cast<float*>(b + L.off[KVC_BUF_K_SCALE]);
  d.v_scale = reinterpret_cast<float*>(b + L.off[KVC_BUF_V_SCALE]);
  d.slot_pos = reinterpret_cast<int32_t*>(b + L.off[KVC_BUF_SLOT_POS]);
  d.score = reinterpret_cast<float*>(b + L.off[KVC_BUF_SCORE]);
  d.sink_k = reinterpret_cast<uint16_t*>(b + L.off[KVC_BUF_SINK_K]);
  d.sink_v = reinterpret_cast<uint16_t*>(b + L.off[KVC_BUF_SINK_V]);
  d.sink_score = reinterpret_cast<float*>(b + L.off[KVC_BUF_SINK_SCORE]);
  d.block_table = reinterpret_cast<int32_t*>(b + L.off[KVC_BUF_BLOCK_TABLE]);
  d.seq_slots = reinterpret_cast<int32_t*>(b + L.off[KVC_BUF_SEQ_SLOTS]);
  d.seq_pos = reinterpret_cast<int32_t*>(b + L.off[KVC_BUF_SEQ_POS]);
  d.free_stack = reinterpret_cast<int32_t*>(b + L.off[KVC_BUF_FREE_STACK]);
  d.counters = reinterpret_cast<int32_t*>(b + L.off[KVC_BUF_COUNTERS]);
  d.plan = reinterpret_cast<int32_t*>(b + L.off[KVC_BUF_PLAN]);
  d.ring_k = reinterpret_cast<uint16_t*>(b + L.off[KVC_BUF_RING_K]);
  d.ring_v = reinterpret_cast<uint16_t*>(b + L.off[KVC_BUF_RING_V]);
  d.ring_score = reinterpret_cast<float*>(b + L.off[KVC_BUF_RING_SCORE]);
  d.ring = cfg->bf16_window;
  d.fp8 = cfg->codes == KVC_CODES_E4M3 ? 1 : 0;
  d.hq = cfg->num_q_heads;
  d.hkv = cfg->num_kv_heads;
  d.group = cfg->num_q_heads / cfg->num_kv_heads;
  d.bits = cfg->bits;
  d.row_bytes = kvc::kHeadDim * cfg->bits / 8;
  d.num_blocks = cfg->num_blocks;
  d.max_batch = cfg->max_batch;
  d.max_bps = cfg->max_blocks_per_seq;
  c->slots.assign(cfg->max_batch, 0);
  c->pos.assign(cfg->max_batch, 0);
  *out = c;
  return KVC_OK;
}

void kvc_cache_destroy(kvc_cache* cache) {
  if (!cache) return;
  // (an event may be destroyed with work pending: it is released once done)
  if (cache->merge_done) cudaEventDestroy(cache->merge_done);
  if (cache->evict_done) cudaEventDestroy(cache->evict_done);
  delete cache;
}

kvc_status kvc_cache_buffer(const kvc_cache* c, int32_t which, void** d_ptr, size_t* bytes) {
  if (!c || which < 0 || which >= KVC_BUF_COUNT) return KVC_ERR_INVALID_ARG;
  if (d_ptr) *d_ptr = c->base + c->layout.off[which];
  if (bytes) *bytes = c->layout.size[which];
  return KVC_OK;
}

kvc_status kvc_cache_lengths(const kvc_cache* c, int32_t seq, int32_t* slots, int32_t* positions) {
  if (!c || seq < 0 || seq >= c->cfg.max_batch) return KVC_ERR_INVALID_ARG;
  if (slots) *slots = c->slots[seq];
  if (positions) *positions = c->pos[seq];
  return KVC_OK;
}

kvc_status kvc_cache_reset(kvc_cache* c, const int32_t* h_block_order, void* stream) {
  if (!c) return KVC_ERR_INVALID_ARG;
  {
    const kvc_status oe = order_after_eviction(c, static_cast<cudaStream_t>(stream));
    if (oe != KVC_OK) return oe;
  }
  const int nb = c->cfg.num_blocks;
  if (h_block_order) {
    std::vector<char> seen(nb, 0);
    for (int i = 0; i < nb; ++i) {
      const int v = h_block_order[i];
      if (v < 0 || v >= nb || seen[v]) return KVC_ERR_INVALID_ARG;
      seen[v] = 1;
    }
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  c->last_launches = 0;
  if (cudaMemsetAsync(c->base, 0, c->layout.total, st) != cudaSuccess) return KVC_ERR_CUDA;
  if (h_block_order) {
    if (cudaMemcpyAsync(c->dev.free_stack, h_block_order, (size_t)nb * 4, cudaMemcpyHostToDevice, st) !=
        cudaSuccess)
      return KVC_ERR_CUDA;
  } else {
    if (kvc::launch_fill_free_stack(c->dev, st) != cudaSuccess) return KVC_ERR_CUDA;
    c->last_launches = 1;
  }
  const int32_t top = nb;
  if (cudaMemcpyAsync(c->dev.counters + kvc::kCtrFreeTop, &top, 4, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return KVC_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return KVC_ERR_CUDA;
  std::fill(c->slots.begin(), c->slots.end(), 0);
  std::fill(c->pos.begin(), c->pos.end(), 0);
  c->plan_pending = false;
  return KVC_OK;
}

kvc_status kvc_release_sequences(kvc_cache* c, int32_t seq_begin, int32_t batch, void* stream) {
  if (!c) return KVC_ERR_INVALID_ARG;
  {
    const kvc_status oe = order_after_eviction(c, static_cast<cudaStream_t>(stream));
    if (oe != KVC_OK) return oe;
  }
  c->last_launches = 0;
  if (!range_ok(c, seq_begin, batch)) return KVC_ERR_INVALID_ARG;
  bool any = false;
  for (int i = 0; i < batch; ++i) any |= c->pos[seq_begin + i] != 0;
  c->plan_pending = false;
  if (!any) return KVC_OK;
  if (kvc::launch_release_sequences(c->dev, seq_begin, batch, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KVC_ERR_CUDA;
  c->last_launches = 1;
  for (int i = 0; i < batch; ++i) {
    c->slots[seq_begin + i] = 0;
    c->pos[seq_begin + i] = 0;
  }
  return KVC_OK;
}

kvc_status kvc_cache_sync_host(kvc_cache* c, void* stream) {
  if (!c) return KVC_ERR_INVALID_ARG;
  {
    const kvc_status oe = order_after_eviction(c, static_cast<cudaStream_t>(stream));
    if (oe != KVC_OK) return oe;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int mb = c->cfg.max_batch;
  std::vector<int32_t> s(mb), p(mb);
  if (cudaMemcpyAsync(s.data(), c->dev.seq_slots, (size_t)mb * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemcpyAsync(p.data(), c->dev.seq_pos, (size_t)mb * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return KVC_ERR_CUDA;
  c->slots = s;
  c->pos = p;
  c->plan_pending = false;
  return KVC_OK;
}

size_t kvc_workspace_bytes(const kvc_cache* c, int32_t batch) {
  if (!c || batch <= 0 || batch > c->cfg.max_batch) return 0;
  return ws_layout(c, batch).total;
}

kvc_status kvc_quantize_append(kvc_cache* c, int32_t seq_begin, int32_t batch, int32_t n_new, const void* d_k,
                               const void* d_v, void* stream) {
  if (!c) return KVC_ERR_INVALID_ARG;
  {
    const kvc_status oe = order_after_eviction(c, static_cast<cudaStream_t>(stream));
    if (oe != KVC_OK) return oe;
  }
  c->last_launches = 0;
  if (!range_ok(c, seq_begin, batch) || n_new < 0) return KVC_ERR_INVALID_ARG;
  if (n_new == 0) return KVC_OK;
  if (!d_k || !d_v || !aligned(d_k, 8) || !aligned(d_v, 8)) return KVC_ERR_INVALID_ARG;
  // capacity, from the host mirror (no device round trip)
  long long need = 0;
  std::vector<int32_t> new_slots(batch);
  for (int i = 0; i < batch; ++i) {
    const int b = seq_begin + i;
    if ((long long)c->pos[b] + n_new > 2000000000LL) return KVC_ERR_CAPACITY;
    int lo, hi;  // positions entering the pool (the device computes the same)
    kvc::pool_range(c->pos[b], n_new, c->cfg.bf16_window, &lo, &hi);
    const long long ns = (long long)c->slots[b] + (hi - lo);
    if ((ns + kvc::kPage - 1) / kvc::kPage > c->cfg.max_blocks_per_seq) return KVC_ERR_CAPACITY;
    need += pages_of((int)ns) - pages_of(c->slots[b]);
    new_slots[i] = (int32_t)ns;
  }
  if (need > (long long)c->cfg.num_blocks - used_pages(c)) return KVC_ERR_CAPACITY;
  // long appends that move no window token into the pool: rows spread over
  // (token chunk, sequence) CTAs, read with 16-byte loads
  bool bulk = n_new >= kvc::kBulkAppendMin && aligned(d_k, 16) && aligned(d_v, 16);
  for (int i = 0; i < batch && bulk; ++i) {
    int lo, hi;
    kvc::pool_range(c->pos[seq_begin + i], n_new, c->cfg.bf16_window, &lo, &hi);
    if (c->cfg.bf16_window > 0 && std::min(c->pos[seq_begin + i], hi) > lo) bulk = false;
  }
  const cudaError_t e =
      bulk ? kvc::launch_append_bulk(c->dev, seq_begin, batch, n_new, static_cast<const uint16_t*>(d_k),
                                     static_cast<const uint16_t*>(d_v), static_cast<cudaStream_t>(stream))
           : kvc::launch_append(c->dev, seq_begin, batch, n_new, static_cast<const uint16_t*>(d_k),
                                static_cast<const uint16_t*>(d_v), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return KVC_ERR_CUDA;
  c->last_launches = bulk ? 2 : 1;
  for (int i = 0; i < batch; ++i) {
    c->slots[seq_begin + i] = new_slots[i];
    c->pos[seq_begin + i] += n_new;
  }
  c->plan_pending = false;
  return KVC_OK;
}

kvc_status kvc_decode_attention(kvc_cache* c, int32_t seq_begin, int32_t batch, const void* d_q, void* d_out,
                                float sm_scale, int32_t flags, void* d_workspace, size_t workspace_bytes,
                                void* stream) {
  if (!c) return KVC_ERR_INVALID_ARG;
  {
    const kvc_status oe = order_after_eviction(c, static_cast<cudaStream_t>(stream));
    if (oe != KVC_OK) return oe;
  }
  c->last_launches = 0;
  if (flags & ~KVC_ATTN_ACCUM_H2O) return KVC_ERR_INVALID_ARG;
  kvc_status st0 = attention_check(c, seq_begin, batch, d_q, d_out, sm_scale, d_workspace, workspace_bytes, 0);
  if (st0 != KVC_OK) return st0;
  kvc::AttnWork w;
  long long total_pages = 0;
  attention_plan(c, seq_begin, batch, d_workspace, &w, &total_pages);
  const float qk_scale_log2 = sm_scale * 1.4426950408889634f;
  const bool h2o = (flags & KVC_ATTN_ACCUM_H2O) != 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int launches = 0;
  // (launched even with no pool pages: its first CTA publishes the page
  // prefix the merge reads)
  st0 = launch_split_traced(c, seq_begin, batch, d_q, qk_scale_log2, w, h2o, total_pages, st, &launches,
                            /*always=*/true);
  if (st0 != KVC_OK) return st0;
  st0 = launch_ring(c, seq_begin, batch, d_q, qk_scale_log2, w, st, &launches);
  if (st0 != KVC_OK) return st0;
  if (kvc::launch_attention_merge(c->dev, seq_begin, batch, static_cast<const uint16_t*>(d_q),
                                  static_cast<uint16_t*>(d_out), qk_scale_log2, w,
                                  h2o ? kvc::kMergeAllScores : kvc::kMergeNoScores, st) != cudaSuccess)
    return KVC_ERR_CUDA;
  ++launches;
  c->last_launches = launches;
  return KVC_OK;
}

kvc_status kvc_h2o_select_evict(kvc_cache* c, int32_t seq_begin, int32_t batch, const kvc_evict_params* p,
                                uint8_t* d_keep_mask, void* d_workspace, size_t workspace_bytes, void* stream) {
  if (!c) return KVC_ERR_INVALID_ARG;
  {
    const kvc_status oe = order_after_eviction(c, static_cast<cudaStream_t>(stream));
    if (oe != KVC_OK) return oe;
  }
  c->last_launches = 0;
  if (!range_ok(c, seq_begin, batch) || !p || !d_keep_mask) return KVC_ERR_INVALID_ARG;
  {
    const kvc_status e = evict_check(c, p);
    if (e != KVC_OK) return e;
  }
  const WsLayout wl = ws_layout(c, batch);
  if (!d_workspace || !aligned(d_workspace, kAlign) || workspace_bytes < wl.total) return KVC_ERR_INVALID_ARG;
  std::vector<int32_t> plan(batch);
  int max_s = 0;
  for (int i = 0; i < batch; ++i) {
    const int b = seq_begin + i;
    const int S = c->slots[b];
    plan[i] = plan_keep(p, S, c->pos[b], c->cfg.bf16_window);
    max_s = std::max(max_s, S);
  }
  if (p->mode == KVC_EVICT_BLOCK) {
    if (c->cfg.max_blocks_per_seq > kvc::kMaxBlockPages) return KVC_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto* keys = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(d_workspace) + wl.keys);
    if (kvc::launch_block_keys(c->dev, seq_begin, batch, p->recent, max_block_cand(c, seq_begin, batch, p->recent), keys,
                               st) != cudaSuccess ||
        kvc::launch_select_blocks(c->dev, seq_begin, batch, p->recent, p->retention, keys, d_keep_mask, s_cap(c),
                                  st) != cudaSuccess)
      return KVC_ERR_CUDA;
    c->last_launches = 2;
    c->plan_pending = true;
    c->plan_block = true;
    c->plan_begin = seq_begin;
    c->plan_batch = batch;
    c->plan_new = plan;
    return KVC_OK;
  }
  uint8_t* ws = static_cast<uint8_t*>(d_workspace);
  kvc::SelectArgs a{};
  a.mode = p->mode;
  a.budget = p->budget;
  a.recent = p->recent;
  a.window = p->window;
  a.s_cap = s_cap(c);
  a.smem_slots = max_s <= kvc::select_max_smem_slots() ? std::max(max_s, 1) : 0;
  a.g_keys = reinterpret_cast<uint32_t*>(ws + wl.keys);
  a.g_pos = reinterpret_cast<int32_t*>(ws + wl.pos);
  if (kvc::launch_select(c->dev, seq_begin, batch, a, d_keep_mask, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return KVC_ERR_CUDA;
  c->last_launches = 1;
  c->plan_pending = true;
  c->plan_block = false;
  c->plan_begin = seq_begin;
  c->plan_batch = batch;
  c->plan_new = plan;
  return KVC_OK;
}

kvc_status kvc_compact_blocks(kvc_cache* c, int32_t seq_begin, int32_t batch, const uint8_t* d_keep_mask,
                              void* d_workspace, size_t workspace_bytes, void* stream) {
  if (!c) return KVC_ERR_INVALID_ARG;
  {
    const kvc_status oe = order_after_eviction(c, static_cast<cudaStream_t>(stream));
    if (oe != KVC_OK) return oe;
  }
  c->last_launches = 0;
  if (!range_ok(c, seq_begin, batch) || !d_keep_mask) return KVC_ERR_INVALID_ARG;
  if (!c->plan_pending || c->plan_begin != seq_begin || c->plan_batch != batch) return KVC_ERR_STATE;
  const WsLayout wl = ws_layout(c, batch);
  if (!d_workspace || !aligned(d_workspace, kAlign) || workspace_bytes < wl.total) return KVC_ERR_INVALID_ARG;
  if (!aligned(d_keep_mask, 16)) return KVC_ERR_INVALID_ARG;
  if (c->plan_block) {
    // block-granular plan: the row drops the pages, nothing moves
    if (kvc::launch_release_blocks(c->dev, seq_begin, batch, d_keep_mask, s_cap(c),
                                   static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return KVC_ERR_CUDA;
    c->last_launches = 1;
    for (int i = 0; i < batch; ++i) c->slots[seq_begin + i] = c->plan_new[i];
    c->plan_pending = false;
    return KVC_OK;
  }
  uint8_t* ws = static_cast<uint8_t*>(d_workspace);
  // largest move count of the slice: min(kept, evicted) per sequence
  int max_moves = 0;
  for (int i = 0; i < batch; ++i) {
    const int S = c->slots[seq_begin + i], np = c->plan_new[i];
    if (np < S) max_moves = std::max(max_moves, std::min(np, S - np));
  }
  const int smem_moves = max_moves <= kvc::compact_max_smem_moves() ? std::max(max_moves, 1) : 0;
  if (kvc::launch_compact(c->dev, seq_begin, batch, d_keep_mask, s_cap(c), reinterpret_cast<int32_t*>(ws + wl.keys),
                          reinterpret_cast<int32_t*>(ws + wl.pos), smem_moves,
                          static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KVC_ERR_CUDA;
  c->last_launches = 2;  // compaction, then the release of the emptied pages
  for (int i = 0; i < batch; ++i) c->slots[seq_begin + i] = c->plan_new[i];
  c->plan_pending = false;
  return KVC_OK;
}

namespace {

kvc_status ensure_events(kvc_cache* c) {
  if (!c->merge_done && cudaEventCreateWithFlags(&c->merge_done, cudaEventDisableTiming) != cudaSuccess)
    return KVC_ERR_CUDA;
  if (!c->evict_done && cudaEventCreateWithFlags(&c->evict_done, cudaEventDisableTiming) != cudaSuccess)
    return KVC_ERR_CUDA;
  return KVC_OK;
}

// The one-call decode step; with `overlap`, the merge runs on `stream` and
// the eviction (scores, selection, compaction) on `evict_stream` after it.
kvc_status decode_step_impl(kvc_cache* c, int32_t seq_begin, int32_t batch, const void* d_q, const void* d_k_new,
                            const void* d_v_new, void* d_out, float sm_scale, const kvc_evict_params* params,
                            void* d_workspace, size_t workspace_bytes, void* stream, void* evict_stream,
                            bool overlap) {
  if (!c) return KVC_ERR_INVALID_ARG;
  c->last_launches = 0;
  {
    const kvc_status e = evict_check(c, params);
    if (e != KVC_OK) return e;
  }
  const bool block = params->mode == KVC_EVICT_BLOCK;
  if (block && c->cfg.max_blocks_per_seq > kvc::kMaxBlockPages) return KVC_ERR_UNSUPPORTED;
  kvc_status st0 =
      attention_check(c, seq_begin, batch, d_q, d_out, sm_scale, d_workspace, workspace_bytes, /*appended=*/1);
  if (st0 != KVC_OK) return st0;
  // append one token to each sequence (checks capacity before anything runs)
  st0 = kvc_quantize_append(c, seq_begin, batch, 1, d_k_new, d_v_new, stream);
  if (st0 != KVC_OK) return st0;
  int launches = c->last_launches;
  kvc::AttnWork w;
  long long total_pages = 0;
  attention_plan(c, seq_begin, batch, d_workspace, &w, &total_pages);
  const float qk_scale_log2 = sm_scale * 1.4426950408889634f;
  const bool h2o = params->mode != KVC_EVICT_STREAMING;  // H2O scores (token or block selection)
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  st0 = launch_split_traced(c, seq_begin, batch, d_q, qk_scale_log2, w, h2o, total_pages, st, &launches,
                            /*always=*/true);
  if (st0 != KVC_OK) return st0;
  st0 = launch_ring(c, seq_begin, batch, d_q, qk_scale_log2, w, st, &launches);
  if (st0 != KVC_OK) return st0;
  // overlap: the merge (outputs, per-head (M, L), sink scores) on `stream`,
  // then the eviction stream waits for it
  cudaStream_t est = st;
  if (overlap) {
    if (ensure_events(c) != KVC_OK) return KVC_ERR_CUDA;
    if (kvc::launch_attention_merge(c->dev, seq_begin, batch, static_cast<const uint16_t*>(d_q),
                                    static_cast<uint16_t*>(d_out), qk_scale_log2, w,
                                    h2o ? kvc::kMergeSinkScores : kvc::kMergeNoScores, st) != cudaSuccess)
      return KVC_ERR_CUDA;
    ++launches;
    est = static_cast<cudaStream_t>(evict_stream);
    if (cudaEventRecord(c->merge_done, st) != cudaSuccess || cudaStreamWaitEvent(est, c->merge_done, 0) != cudaSuccess)
      return KVC_ERR_CUDA;
  }
  std::vector<int32_t> plan(batch);
  int max_s = 0;
  for (int i = 0; i < batch; ++i) {
    const int b = seq_begin + i;
    plan[i] = plan_keep(params, c->slots[b], c->pos[b], c->cfg.bf16_window);
    max_s = std::max(max_s, c->slots[b]);
  }
  const WsLayout wl = ws_layout(c, batch);
  uint8_t* ws = static_cast<uint8_t*>(d_workspace);
  kvc::StepArgs a{};
  a.mode = params->mode;
  a.budget = params->budget;
  a.recent = params->recent;
  a.window = params->window;
  a.s_cap = s_cap(c);
  // the score pass writes whole quarter pages of keys; keys and positions in
  // shared memory when both fit, else the keys alone, else neither
  const int slots4 = std::max((max_s + 3) & ~3, 4);
  if (block) {  // no slot keys: the page selection follows
    a.smem_slots = 0;
    a.pos_smem = 0;
  } else if (slots4 * 8 <= kvc::step_max_smem_bytes()) {
    a.smem_slots = slots4;
    a.pos_smem = 1;
  } else if (slots4 * 4 <= kvc::step_max_smem_bytes()) {
    a.smem_slots = slots4;
    a.pos_smem = 0;
  } else {
    a.smem_slots = 0;
    a.pos_smem = 0;
  }
  a.g_keys = reinterpret_cast<uint32_t*>(ws + wl.keys);
  a.g_pos = reinterpret_cast<int32_t*>(ws + wl.pos);
  a.n_moves = reinterpret_cast<int*>(ws + wl.moves);
  int max_moves = 0;  // a pair moves at most min(n', S - n') rows
  for (int i = 0; i < batch; ++i)
    max_moves = std::max(max_moves, std::min(plan[i], c->slots[seq_begin + i] - plan[i]));
  a.inline_moves = !block && max_moves <= kvc::kInlineMoves;
  a.merged = overlap ? 1 : 0;
  if (kvc::launch_step_post(c->dev, seq_begin, batch, static_cast<const uint16_t*>(d_q),
                            static_cast<uint16_t*>(d_out), qk_scale_log2, w, a, sm_count(c), est) != cudaSuccess)
    return KVC_ERR_CUDA;
  ++launches;
  if (block) {
    // page keys over the whole GPU, then one CTA per sequence selects and
    // drops its pages (no rows move)
    auto* keys = reinterpret_cast<unsigned long long*>(ws + wl.keys);
    if (kvc::launch_block_keys(c->dev, seq_begin, batch, params->recent,
                               max_block_cand(c, seq_begin, batch, params->recent), keys, est) != cudaSuccess ||
        kvc::launch_evict_blocks(c->dev, seq_begin, batch, params->recent, params->retention, keys, est) !=
            cudaSuccess)
      return KVC_ERR_CUDA;
    launches += 2;
  } else if (!a.inline_moves) {
    if (kvc::launch_step_moves(c->dev, batch, a, sm_count(c), max_moves, est) != cudaSuccess) return KVC_ERR_CUDA;
    ++launches;
  }
  if (overlap) {
    // later calls on this cache order themselves after this event
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    unsigned long long id = 0;
    if (cudaEventRecord(c->evict_done, est) != cudaSuccess || cudaStreamGetCaptureInfo(est, &cs, &id) != cudaSuccess)
      return KVC_ERR_CUDA;
    c->evict_pending = true;
    c->evict_in_capture = cs == cudaStreamCaptureStatusActive;
    c->evict_capture_id = id;
  }
  for (int i = 0; i < batch; ++i) c->slots[seq_begin + i] = plan[i];
  c->plan_pending = false;
  c->last_launches = launches;
  return KVC_OK;
}

}  // namespace

kvc_status kvc_decode_step(kvc_cache* c, int32_t seq_begin, int32_t batch, const void* d_q, const void* d_k_new,
                           const void* d_v_new, void* d_out, float sm_scale, const kvc_evict_params* params,
                           void* d_workspace, size_t workspace_bytes, void* stream) {
  return decode_step_impl(c, seq_begin, batch, d_q, d_k_new, d_v_new, d_out, sm_scale, params, d_workspace,
                          workspace_bytes, stream, stream, false);
}

kvc_status kvc_decode_step_overlap(kvc_cache* c, int32_t seq_begin, int32_t batch, const void* d_q,
                                   const void* d_k_new, const void* d_v_new, void* d_out, float sm_scale,
                                   const kvc_evict_params* params, void* d_workspace, size_t workspace_bytes,
                                   void* stream, void* evict_stream) {
  return decode_step_impl(c, seq_begin, batch, d_q, d_k_new, d_v_new, d_out, sm_scale, params, d_workspace,
                          workspace_bytes, stream, evict_stream, true);
}

size_t kvc_prefill_workspace_bytes(const kvc_cache* c, int32_t batch, int32_t n) {
  if (!c || batch <= 0 || n <= 0) return 0;
  return align_up((size_t)batch * c->cfg.num_q_heads * n * 2 * 4);
}

kvc_status kvc_prefill_attention(kvc_cache* c, int32_t seq_begin, int32_t batch, int32_t n, const void* d_q,
                                 const void* d_k, const void* d_v, void* d_out, float sm_scale, int32_t flags,
                                 void* d_workspace, size_t workspace_bytes, void* stream) {
  if (!c) return KVC_ERR_INVALID_ARG;
  {
    const kvc_status oe = order_after_eviction(c, static_cast<cudaStream_t>(stream));
    if (oe != KVC_OK) return oe;
  }
  c->last_launches = 0;
  if (!range_ok(c, seq_begin, batch) || n <= 0 || (flags & ~KVC_ATTN_ACCUM_H2O)) return KVC_ERR_INVALID_ARG;
  if (!d_q || !d_out || !aligned(d_q, 16) || !aligned(d_out, 16) || !d_k || !d_v || !aligned(d_k, 16) ||
      !aligned(d_v, 16))
    return KVC_ERR_INVALID_ARG;
  if (!(sm_scale > 0.0f) || !std::isfinite(sm_scale)) return KVC_ERR_INVALID_ARG;
  if (!d_workspace || !aligned(d_workspace, kAlign) ||
      workspace_bytes < kvc_prefill_workspace_bytes(c, batch, n))
    return KVC_ERR_INVALID_ARG;
  if ((long long)n * kvc::kHeadDim * c->cfg.num_q_heads * batch > 2000000000000LL) return KVC_ERR_UNSUPPORTED;
  for (int i = 0; i < batch; ++i)
    if (c->pos[seq_begin + i] != 0) return KVC_ERR_STATE;  // a prompt starts a sequence
  kvc_status st0 = kvc_quantize_append(c, seq_begin, batch, n, d_k, d_v, stream);
  if (st0 != KVC_OK) return st0;
  const bool h2o = (flags & KVC_ATTN_ACCUM_H2O) != 0;
  if (kvc::launch_prefill(c->dev, seq_begin, batch, n, static_cast<const uint16_t*>(d_q),
                          static_cast<const uint16_t*>(d_k), static_cast<const uint16_t*>(d_v),
                          static_cast<uint16_t*>(d_out), static_cast<float*>(d_workspace),
                          sm_scale * 1.4426950408889634f, h2o, static_cast<cudaStream_t>(stream),
                          static_cast<cudaEvent_t>(c->trace_start && c->trace_stop ? c->trace_start : nullptr),
                          static_cast<cudaEvent_t>(c->trace_start && c->trace_stop ? c->trace_stop : nullptr)) !=
      cudaSuccess)
    return KVC_ERR_CUDA;
  c->last_launches += 1 + (h2o ? 1 : 0);
  return KVC_OK;
}

// Workspace of kvc_prefill_context: per (sequence, KV head) the row
// statistics of its n * G attention rows, one row of column sums per CTA of
// the multi-query kernel (sinks first, then every pool slot, then the bf16
// window's positions), a ticket.
struct CtxWs {
  size_t stats, colsum, ticket, total;
};
CtxWs ctx_ws(const kvc_cache* c, int32_t batch, int32_t n) {
  const size_t pairs = (size_t)batch * c->cfg.num_kv_heads;
  const int G = c->cfg.num_q_heads / c->cfg.num_kv_heads;
  CtxWs w;
  w.stats = 0;
  w.colsum = align_up(pairs * n * G * 2 * 4);
  w.ticket = w.colsum + align_up(pairs * kvc::ctx_groups(n, G) *
                                 (kvc::kSinks + (size_t)s_cap(c) + c->cfg.bf16_window) * 4);
  w.total = w.ticket + align_up(pairs * 4);
  return w;
}

size_t kvc_prefill_context_workspace_bytes(const kvc_cache* c, int32_t batch, int32_t n) {
  if (!c || batch <= 0 || n <= 0) return 0;
  return ctx_ws(c, batch, n).total;
}

kvc_status kvc_prefill_context(kvc_cache* c, int32_t seq_begin, int32_t batch, int32_t n, const void* d_q,
                               const void* d_k, const void* d_v, void* d_out, float sm_scale, int32_t flags,
                               void* d_workspace, size_t workspace_bytes, void* stream) {
  if (!c) return KVC_ERR_INVALID_ARG;
  {
    const kvc_status oe = order_after_eviction(c, static_cast<cudaStream_t>(stream));
    if (oe != KVC_OK) return oe;
  }
  c->last_launches = 0;
  if (!range_ok(c, seq_begin, batch) || n <= 0 || (flags & ~KVC_ATTN_ACCUM_H2O)) return KVC_ERR_INVALID_ARG;
  if (!d_q || !d_out || !aligned(d_q, 16) || !aligned(d_out, 16) || !d_k || !d_v || !aligned(d_k, 16) ||
      !aligned(d_v, 16))
    return KVC_ERR_INVALID_ARG;
  if (!(sm_scale > 0.0f) || !std::isfinite(sm_scale)) return KVC_ERR_INVALID_ARG;
  if (!d_workspace || !aligned(d_workspace, kAlign) ||
      workspace_bytes < kvc_prefill_context_workspace_bytes(c, batch, n))
    return KVC_ERR_INVALID_ARG;
  if ((long long)n * c->cfg.num_q_heads > (1LL << 30)) return KVC_ERR_UNSUPPORTED;
  kvc_status st0 = kvc_quantize_append(c, seq_begin, batch, n, d_k, d_v, stream);
  if (st0 != KVC_OK) return st0;
  int launches = c->last_launches;
  const CtxWs wl = ctx_ws(c, batch, n);
  uint8_t* ws = static_cast<uint8_t*>(d_workspace);
  if (kvc::launch_ctx_attention(c->dev, seq_begin, batch, n, static_cast<const uint16_t*>(d_q),
                                static_cast<uint16_t*>(d_out), reinterpret_cast<float*>(ws + wl.stats),
                                reinterpret_cast<float*>(ws + wl.colsum), reinterpret_cast<int*>(ws + wl.ticket),
                                s_cap(c), sm_scale * 1.4426950408889634f, (flags & KVC_ATTN_ACCUM_H2O) != 0,
                                static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    c->last_launches = launches;
    return KVC_ERR_CUDA;
  }
  c->last_launches = launches + 2;
  return KVC_OK;
}

kvc_status kvc_read_status(kvc_cache* c, int32_t* h_status, void* stream) {
  if (!c || !h_status) return KVC_ERR_INVALID_ARG;
  {
    const kvc_status oe = order_after_eviction(c, static_cast<cudaStream_t>(stream));
    if (oe != KVC_OK) return oe;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, c->dev.counters + kvc::kCtrStatus, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return KVC_ERR_CUDA;
  *h_status = v;
  if (v != 0) {
    if (cudaMemsetAsync(c->dev.counters + kvc::kCtrStatus, 0, 4, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return KVC_ERR_CUDA;
    return KVC_ERR_DEVICE;
  }
  return KVC_OK;
}

kvc_status kvc_set_trace_events(kvc_cache* c, void* ev_start, void* ev_stop) {
  if (!c || ((ev_start == nullptr) != (ev_stop == nullptr))) return KVC_ERR_INVALID_ARG;
  c->trace_start = ev_start;
  c->trace_stop = ev_stop;
  return KVC_OK;
}

int32_t kvc_last_launch_count(const kvc_cache* c) { return c ? c->last_launches : 0; }

}  // extern "C"
