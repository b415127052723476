// Kept-set selection and compaction of the paged pool.
//
// Selection ("KV Cache optimization techniques" sections 2.2 and 2.4;
// Technical Report sections 3.3 and 3.4): per (sequence, KV head), keep the
// recent window and the top-k of the other slots by accumulated H2O score,
// ties to the lower position, or, in StreamingLLM mode, exactly the last
// `window` positions.  The sinks live outside the pool and are always kept.
//
// GB300 design: one CTA per (KV head, sequence).  Each slot gets a 32-bit key,
// 0xFFFFFFFF for the recent window (always kept) and the fp32 score's bit
// pattern otherwise (scores are >= 0, so the bit patterns order like the
// values).  The n_keep-th largest key is found by an MSB-first radix select
// (four 8-bit passes, shared-memory histograms); ties at the threshold key are
// resolved by a second radix select on the positions (smallest first).  Keys
// and positions sit in shared memory when they fit, else in the workspace.
//
// Compaction: with n' kept slots, the evicted slots below n' ("holes") are
// filled in ascending order by the kept slots at or above n' (ascending).
// Sources all lie at or above n' and destinations below it, so the moves never
// overlap.  The pages past ceil(n'/16) go back to the free-block stack.
#include "kvc_device.h"
#include "kvc_internal.h"

namespace kvc {
namespace {

using namespace dev;

constexpr int kSelThreads = 1024;
constexpr int kCompactThreads = 512;
constexpr int kSelBtStage = 2048;  // block-table entries staged in shared memory


__global__ void __launch_bounds__(kSelThreads) select_kernel(DevState s, int seq_begin, SelectArgs a,
                                                            uint8_t* __restrict__ mask) {
  const int h = blockIdx.x;
  const int bl = blockIdx.y;
  const int b = seq_begin + bl;
  const int S = s.seq_slots[b];
  const int P = s.seq_pos[b];
  const int ns = min(P, kSinks);
  uint8_t* mrow = mask + ((size_t)bl * s.hkv + h) * a.s_cap;
  bool keep_all;
  int n_keep, thr;
  if (a.mode == 0) {
    keep_all = ns + S <= a.budget;
    n_keep = a.budget - kSinks;
    thr = P - a.recent;
  } else {
    keep_all = S <= a.window;
    n_keep = a.window;
    thr = P - a.window;
  }
  if (keep_all) n_keep = S;
  if (h == 0 && threadIdx.x == 0) {
    s.plan[2 * b] = S;
    s.plan[2 * b + 1] = n_keep;
  }
  if (keep_all || n_keep <= 0) {
    for (int t = threadIdx.x; t < S; t += blockDim.x) mrow[t] = keep_all ? 1 : 0;
    return;
  }

  extern __shared__ __align__(16) uint32_t dyn[];
  __shared__ int hist[kRadixBins];
  __shared__ int sh_sel[3];
  __shared__ int sh_warp[32];
  uint32_t* keys;
  int32_t* pos;
  if (a.smem_slots > 0) {
    keys = dyn;
    pos = reinterpret_cast<int32_t*>(dyn + a.smem_slots);
  } else {
    keys = a.g_keys + ((size_t)bl * s.hkv + h) * a.s_cap;
    pos = a.g_pos + ((size_t)bl * s.hkv + h) * a.s_cap;
  }
  const int32_t* bt = s.block_table + (size_t)b * s.max_bps;
  const bool h2o = a.mode == 0;
  // stage the block-table row in shared memory when it fits
  __shared__ int32_t sh_bt[kSelBtStage];
  const int npages = (S + kPage - 1) / kPage;
  const int32_t* btp = bt;
  if (npages <= kSelBtStage) {
    for (int i = threadIdx.x; i < npages; i += blockDim.x) sh_bt[i] = bt[i];
    btp = sh_bt;
  }
  __syncthreads();
  const int nt = blockDim.x;
  for (int t0 = threadIdx.x; t0 < S; t0 += 4 * nt) {
    int p[4];
    float sc[4];
    bool ok[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = t0 + u * nt;
      const int blk = t < S ? btp[t / kPage] : 0;
      ok[u] = t < S && (unsigned)blk < (unsigned)s.num_blocks;
      const size_t idx = ((size_t)(ok[u] ? blk : 0) * s.hkv + h) * kPage + (t % kPage);
      p[u] = ok[u] ? s.slot_pos[idx] : -1;
      sc[u] = (ok[u] && h2o) ? s.score[idx] : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = t0 + u * nt;
      if (t >= S) continue;
      uint32_t key = 0;
      if (!ok[u]) {
        atomicOr(&s.counters[kCtrStatus], kDevBadBlockId);
      } else if (p[u] >= thr) {
        key = 0xFFFFFFFFu;
      } else if (h2o) {
        key = __float_as_uint(fmaxf(sc[u], 0.0f));
      }
      keys[t] = key;
      pos[t] = p[u];
    }
  }
  __syncthreads();

  int need, ties;
  const uint32_t theta = radix_select<kSelThreads>(
      S, n_keep, true, [&](int) { return true; }, [&](int i) { return keys[i]; }, hist, sh_warp, sh_sel, &need,
      &ties);
  uint32_t pos_cut = 0xFFFFFFFFu;
  if (ties > need) {  // ties at theta: the lowest positions win
    int rem2, t2;
    pos_cut = radix_select<kSelThreads>(
        S, need, false, [&](int i) { return keys[i] == theta; }, [&](int i) { return (uint32_t)pos[i]; }, hist,
        sh_warp, sh_sel, &rem2, &t2);
  }
  for (int t = threadIdx.x; t < S; t += blockDim.x) {
    const uint32_t k = keys[t];
    mrow[t] = (k > theta || (k == theta && (uint32_t)pos[t] <= pos_cut)) ? 1 : 0;
  }
}

// Compaction of one (KV head, sequence).  Phase 1 (tiles of 16 slots per
// thread): the keep-mask bytes of a thread's 16 slots come in one 16-byte
// load; block scans give every hole (evicted slot inside the keep window,
// see keep_window) and every source (kept slot outside it) its rank, and the
// physical pool index of the i-th hole and of the i-th source go to two
// lists.  Phase 2: the row moves
// (move_rows: the lanes of a row store its 16-byte chunks together).
__global__ void __launch_bounds__(kCompactThreads, 2) compact_kernel(DevState s, int seq_begin,
                                                                 const uint8_t* __restrict__ mask, int s_cap,
                                                                 int32_t* __restrict__ g_holes,
                                                                 int32_t* __restrict__ g_srcs, int smem_moves) {
  const int h = blockIdx.x;
  const int bl = blockIdx.y;
  const int b = seq_begin + bl;
  const int S = s.plan[2 * b];
  const int np = s.plan[2 * b + 1];
  if (np >= S) return;
  __shared__ int sh_warp[32];
  extern __shared__ __align__(16) int32_t dyn_lists[];
  const size_t pair = (size_t)bl * s.hkv + h;
  const uint8_t* mrow = mask + pair * s_cap;
  int32_t* holes = smem_moves > 0 ? dyn_lists : g_holes + pair * s_cap;
  int32_t* srcs = smem_moves > 0 ? dyn_lists + smem_moves : g_srcs + pair * s_cap;
  const int32_t* bt = s.block_table + (size_t)b * s.max_bps;
  const int hkv = s.hkv;
  // the sequence's block-table row, staged in shared memory when it fits
  __shared__ int32_t sh_bt[kSelBtStage];
  const int npages = (S + kPage - 1) / kPage;
  const int32_t* btp = bt;
  if (npages <= kSelBtStage) {
    for (int i = threadIdx.x; i < npages; i += blockDim.x) sh_bt[i] = bt[i];
    btp = sh_bt;
  }
  __syncthreads();

  const int wlo = keep_window(S, np);
  int hole_base = 0, src_base = 0;
  for (int tile0 = 0; tile0 < S; tile0 += kCompactThreads * 16) {
    const int t0 = tile0 + threadIdx.x * 16;
    uint32_t kept_bits = 0;
    if (t0 < S) {
      const uint4 m = *reinterpret_cast<const uint4*>(mrow + t0);
      const uint32_t wv[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (((wv[i >> 2] >> (8 * (i & 3))) & 0xFFu) != 0 && t0 + i < S) kept_bits |= 1u << i;
    }
    // bit i of `inwin` is set when slot t0 + i lies in the window [wlo, wlo + n')
    const int lo = min(max(wlo - t0, 0), 16), hi = min(max(wlo + np - t0, 0), 16);
    const uint32_t inwin = ((1u << hi) - 1u) & ~((1u << lo) - 1u);
    const int nv = min(max(S - t0, 0), 16);
    const uint32_t valid = nv >= 16 ? 0xFFFFu : ((1u << nv) - 1u);
    const uint32_t hole_bits = ~kept_bits & inwin & valid;
    const uint32_t src_bits = kept_bits & ~inwin;
    // one scan of both counts (each <= 16 per thread, <= 8192 per tile)
    const int nh = __popc(hole_bits), ns = __popc(src_bits);
    int tot_packed;
    const int incl = block_scan<kCompactThreads>(nh | (ns << 16), sh_warp, &tot_packed);
    int ph = hole_base + (incl & 0xFFFF) - nh;
    int ps = src_base + (incl >> 16) - ns;
    for (uint32_t m = hole_bits; m; m &= m - 1) {
      const int t = t0 + __ffs(m) - 1;
      holes[ph++] = (btp[t / kPage] * hkv + h) * kPage + (t % kPage);
    }
    for (uint32_t m = src_bits; m; m &= m - 1) {
      const int t = t0 + __ffs(m) - 1;
      srcs[ps++] = (btp[t / kPage] * hkv + h) * kPage + (t % kPage);
    }
    hole_base += tot_packed & 0xFFFF;
    src_base += tot_packed >> 16;
  }
  // kept slots = (n' - holes) below n' plus the sources above it; the mask
  // holds exactly n' kept slots iff holes and sources pair up
  if (hole_base != src_base) {
    if (threadIdx.x == 0) atomicOr(&s.counters[kCtrStatus], kDevBadKeepMask);
    return;
  }
  __syncthreads();

  // phase 2: the row moves
  const int n_moves = hole_base;
  move_rows(s, holes, srcs, n_moves);
}

// Release of one sequence's pages after its compaction (one CTA per
// sequence, after every KV head's compact CTA): pages [0, p0) and
// [p0 + ceil(n'/16), ceil(S/16)) go to the free stack, the row drops its
// first p0 = w / 16 pages (see keep_window) and the sequence holds n' slots.
__global__ void __launch_bounds__(256) release_kernel(DevState s, int seq_begin) {
  const int b = seq_begin + blockIdx.x;
  const int S = s.plan[2 * b];
  const int np = s.plan[2 * b + 1];
  if (np >= S) return;
  const int keep_pages = (np + kPage - 1) / kPage;
  const int old_pages = (S + kPage - 1) / kPage;
  const int nfree = old_pages - keep_pages;
  const int p0 = keep_window(S, np) / kPage;
  int32_t* row = s.block_table + (size_t)b * s.max_bps;
  __shared__ int sh_base;
  if (threadIdx.x == 0) {
    int base = -1;
    if (nfree > 0) {
      base = atomicAdd(&s.counters[kCtrFreeTop], nfree);
      if (base + nfree > s.num_blocks) {
        atomicSub(&s.counters[kCtrFreeTop], nfree);
        atomicOr(&s.counters[kCtrStatus], kDevStackOverflow);
        base = -1;
      }
    }
    sh_base = base;
    s.seq_slots[b] = np;
  }
  __syncthreads();
  if (sh_base >= 0)
    for (int j = threadIdx.x; j < nfree; j += blockDim.x) s.free_stack[sh_base + j] = row[j < p0 ? j : keep_pages + j];
  if (p0 > 0) shift_row(row, p0, keep_pages);
}

// Block-granular eviction (the eviction-and-reuse survey page, section 4:
// the block manager's eviction by attention sorts blocks by the mean
// attention score of their tokens and evicts the first int(n * (1 - ratio))).
// A block is one page of the sequence, shared by every KV head; the
// candidates are the full pages before the last `recent` slots; a page is
// ordered by the fp64 sum of its 16 x Hkv scores, added head by head and slot
// by slot (the sum orders pages as the mean does); ties go to the earlier
// page.  One CTA per sequence: the plan, then the keep mask of every head
// (all heads the same).  The lowest pages are found by radix select on the
// sum's bit pattern (sums are >= 0, so their bits order like their values):
// the high word, then the low word among equal high words, then the page
// index among equal sums.
constexpr int kBlockThreads = 256;

__global__ void __launch_bounds__(kBlockThreads) block_select_kernel(DevState s, int seq_begin, int recent,
                                                                     double retention, uint8_t* __restrict__ mask,
                                                                     int s_cap) {
  __shared__ unsigned long long key[kMaxBlockPages];
  __shared__ int hist[kRadixBins];
  __shared__ int sh_sel[3];
  __shared__ int sh_warp[32];
  const int bl = blockIdx.x;
  const int b = seq_begin + bl;
  const int S = s.seq_slots[b];
  const int hkv = s.hkv;
  const int n_cand = max(0, S - recent) / kPage;
  const int n_evict = (int)((double)n_cand * (1.0 - retention));
  if (threadIdx.x == 0) {
    s.plan[2 * b] = S;
    s.plan[2 * b + 1] = S - kPage * n_evict;
  }
  const int32_t* bt = s.block_table + (size_t)b * s.max_bps;
  for (int p = threadIdx.x; p < n_cand; p += blockDim.x) {
    const int blk = bt[p];
    double acc = 0.0;
    if ((unsigned)blk < (unsigned)s.num_blocks) {
      const float* sc = s.score + (size_t)blk * hkv * kPage;
      for (int i = 0; i < hkv * kPage; ++i) acc += (double)sc[i];  // head by head, slot by slot
    } else {
      atomicOr(&s.counters[kCtrStatus], kDevBadBlockId);
    }
    key[p] = (unsigned long long)__double_as_longlong(acc);
  }
  __syncthreads();
  unsigned long long theta = 0;
  uint32_t idx_cut = 0;
  bool any = n_evict > 0;
  if (any) {
    int need, ties;
    const uint32_t hi = radix_select<kBlockThreads>(
        n_cand, n_evict, false, [&](int) { return true; }, [&](int i) { return (uint32_t)(key[i] >> 32); },
        hist, sh_warp, sh_sel, &need, &ties);
    int need2, ties2;
    const uint32_t lo = radix_select<kBlockThreads>(
        n_cand, need, false, [&](int i) { return (uint32_t)(key[i] >> 32) == hi; },
        [&](int i) { return (uint32_t)key[i]; }, hist, sh_warp, sh_sel, &need2, &ties2);
    theta = ((unsigned long long)hi << 32) | lo;
    int r3, t3;
    idx_cut = radix_select<kBlockThreads>(
        n_cand, need2, false, [&](int i) { return key[i] == theta; }, [&](int i) { return (uint32_t)i; }, hist,
        sh_warp, sh_sel, &r3, &t3);
  }
  // keep mask of every head: a slot goes when its page goes
  for (int h = 0; h < hkv; ++h) {
    uint8_t* mrow = mask + ((size_t)bl * hkv + h) * s_cap;
    for (int t = threadIdx.x; t < S; t += blockDim.x) {
      const int p = t / kPage;
      bool gone = false;
      if (any && p < n_cand) gone = key[p] < theta || (key[p] == theta && (uint32_t)p <= idx_cut);
      mrow[t] = gone ? 0 : 1;
    }
  }
}

// The block-table rewrite of block-granular eviction (one CTA per sequence):
// the pages whose slots the mask drops (head 0's row; every head's is the
// same) leave the row, the others keep their order, the dropped pages go to
// the free stack and the sequence holds S - 16 * dropped slots.  Nothing
// moves in the pool.
__global__ void __launch_bounds__(kBlockThreads) block_release_kernel(DevState s, int seq_begin,
                                                                      const uint8_t* __restrict__ mask,
                                                                      int s_cap) {
  __shared__ int32_t row_in[kMaxBlockPages];
  __shared__ int sh_warp[32];
  __shared__ int sh_base;
  const int bl = blockIdx.x;
  const int b = seq_begin + bl;
  const int S = s.plan[2 * b];
  const int np = s.plan[2 * b + 1];
  if (np >= S) return;
  const int npages = (S + kPage - 1) / kPage;
  int32_t* row = s.block_table + (size_t)b * s.max_bps;
  const uint8_t* m0 = mask + (size_t)bl * s.hkv * s_cap;  // head 0
  for (int p = threadIdx.x; p < npages; p += blockDim.x) row_in[p] = row[p];
  __syncthreads();
  // ranks of kept and dropped pages, chunk by chunk
  int kept_base = 0, drop_base = 0;
  const int n_drop = (S - np) / kPage;
  if (threadIdx.x == 0) {
    int base = -1;
    if (n_drop > 0) {
      base = atomicAdd(&s.counters[kCtrFreeTop], n_drop);
      if (base + n_drop > s.num_blocks) {
        atomicSub(&s.counters[kCtrFreeTop], n_drop);
        atomicOr(&s.counters[kCtrStatus], kDevStackOverflow);
        base = -1;
      }
    }
    sh_base = base;
  }
  for (int c0 = 0; c0 < npages; c0 += kBlockThreads) {
    const int p = c0 + (int)threadIdx.x;
    const bool valid = p < npages;
    const bool keep = valid && m0[p * kPage] != 0;
    const bool drop = valid && !keep;
    int tot;
    const int incl = block_scan<kBlockThreads>((keep ? 1 : 0) | (drop ? 1 << 16 : 0), sh_warp, &tot);
    const int k_rank = kept_base + (incl & 0xFFFF) - (keep ? 1 : 0);
    const int d_rank = drop_base + (incl >> 16) - (drop ? 1 : 0);
    if (keep) row[k_rank] = row_in[p];
    if (drop && sh_base >= 0 && d_rank < n_drop) s.free_stack[sh_base + d_rank] = row_in[p];
    kept_base += tot & 0xFFFF;
    drop_base += tot >> 16;
  }
  if (threadIdx.x == 0) {
    if (drop_base != n_drop) atomicOr(&s.counters[kCtrStatus], kDevBadKeepMask);
    s.seq_slots[b] = np;
  }
}

}  // namespace

int select_max_smem_slots() { return (200 * 1024) / 8; }

cudaError_t launch_select(const DevState& s, int seq_begin, int batch, const SelectArgs& a, uint8_t* keep_mask,
                          cudaStream_t st) {
  const int smem = a.smem_slots > 0 ? a.smem_slots * 8 : 0;
  if (smem > 0) {
    static int done[64] = {0};
    const cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(select_kernel), select_max_smem_slots() * 8, done);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(s.hkv, batch);
  select_kernel<<<grid, kSelThreads, smem, st>>>(s, seq_begin, a, keep_mask);
  return cudaGetLastError();
}

int compact_max_smem_moves() { return (96 * 1024) / 8; }

cudaError_t launch_compact(const DevState& s, int seq_begin, int batch, const uint8_t* keep_mask, int s_cap,
                           int32_t* g_holes, int32_t* g_srcs, int smem_moves, cudaStream_t st) {
  const int smem = smem_moves > 0 ? smem_moves * 8 : 0;
  if (smem > 0) {
    static int done[64] = {0};
    const cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(compact_kernel), compact_max_smem_moves() * 8, done);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(s.hkv, batch);
  compact_kernel<<<grid, kCompactThreads, smem, st>>>(s, seq_begin, keep_mask, s_cap, g_holes, g_srcs, smem_moves);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  release_kernel<<<batch, 256, 0, st>>>(s, seq_begin);
  return cudaGetLastError();
}

cudaError_t launch_select_blocks(const DevState& s, int seq_begin, int batch, int recent, double retention,
                                 uint8_t* keep_mask, int s_cap, cudaStream_t st) {
  block_select_kernel<<<batch, kBlockThreads, 0, st>>>(s, seq_begin, recent, retention, keep_mask, s_cap);
  return cudaGetLastError();
}

cudaError_t launch_release_blocks(const DevState& s, int seq_begin, int batch, const uint8_t* keep_mask,
                                  int s_cap, cudaStream_t st) {
  block_release_kernel<<<batch, kBlockThreads, 0, st>>>(s, seq_begin, keep_mask, s_cap);
  return cudaGetLastError();
}

}  // namespace kvc
