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
// (passes of 11, 11 and 10 bits, shared-memory histograms); ties at the threshold key are
// resolved by a second radix select on the positions (smallest first).  Keys
// and positions sit in shared memory when they fit, else in the workspace.
//
// Compaction into a keep window: with S slots and n' < S kept, the kept slots
// end up in [w, w + n'), w = 16 * floor((S - n') / 16), the last page-aligned
// window of n' slots.  The evicted slots inside the window ("holes") are
// filled in ascending order by the kept slots outside it ("sources",
// ascending); a hole and a source are never the same slot, so the moves never
// overlap.  The w / 16 pages before the window go back to the free-block
// stack and the block-table row drops them.  After a long context the always
// kept recent tokens already sit inside the window and do not move; at steady
// state (one slot evicted) w = 0 and at most one row moves.
#include <algorithm>

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
  // the nr tokens of the bf16 window (hybrid precision) are kept and count
  // inside the budget or window; the choice is among the pool slots
  const int nr = ring_count(P, s.ring);
  if (a.mode == 0) {
    keep_all = ns + nr + S <= a.budget;
    n_keep = a.budget - kSinks - nr;
    thr = P - a.recent;
  } else {
    keep_all = nr + S <= a.window;
    n_keep = a.window - nr;
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
  if (a.smem_slots > 0 && S > a.smem_slots) {
    // the shared key buffer was sized from the host's mirror of the lengths,
    // which is behind the device (state restored without a host resync):
    // flag it and keep every slot
    for (int t = threadIdx.x; t < S; t += blockDim.x) mrow[t] = 1;
    if (threadIdx.x == 0) atomicOr(&s.counters[kCtrStatus], kDevStaleHost);
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
      holes[ph++] = slot_index(s, btp, t, h);
    }
    for (uint32_t m = src_bits; m; m &= m - 1) {
      const int t = t0 + __ffs(m) - 1;
      srcs[ps++] = slot_index(s, btp, t, h);
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
// page.
//
// block_key_kernel: one thread per candidate page (grid-stride over the
// sequence's pages, so any grid is correct for any lengths) writes the sum's
// bit pattern to the workspace.  The sum is one chain of 16 x Hkv dependent
// fp64 additions, each after an fp32 -> fp64 conversion, and both run on
// GB300's narrow fp64 pipe (measured: about 1.6 additions per clock per SM
// at best), so this kernel is bound by that pipe, not by its 512 bytes of
// loads per page; the pages go one per thread in 64-thread CTAs, spread
// over every SM.
//
// block_evict_kernel: one CTA per sequence.  The lowest n_evict keys (sums are
// >= 0, so their bit patterns order like their values) by an MSB-first radix
// select over the 64-bit keys, eight 8-bit passes; among the pages equal to
// the threshold on the selected bits the earliest go first (a block scan in
// page order).  kRelease = false writes the plan and the keep mask of every
// head (all heads the same); kRelease = true applies the eviction at once:
// the dropped pages leave the row (the others keep their order) and go to the
// free stack, and the sequence holds S - 16 * n_evict slots.  Nothing moves in
// the pool.
constexpr int kBlockThreads = 256;
constexpr int kKeyThreads = 64;
constexpr int kEvictThreads = 512;

__global__ void __launch_bounds__(kKeyThreads) block_key_kernel(DevState s, int seq_begin, int recent,
                                                                unsigned long long* __restrict__ keys) {
  const int bl = blockIdx.y;
  const int b = seq_begin + bl;
  const int S = s.seq_slots[b];
  const int n_cand = max(0, S - recent) / kPage;
  const int hkv = s.hkv;
  const int32_t* bt = s.block_table + (size_t)b * s.max_bps;
  unsigned long long* krow = keys + (size_t)bl * s.max_bps;
  for (int p = blockIdx.x * kKeyThreads + threadIdx.x; p < n_cand; p += gridDim.x * kKeyThreads) {
    const int blk = bt[p];
    double acc = 0.0;
    if ((unsigned)blk < (unsigned)s.num_blocks) {
      // the page's scores are contiguous: [head][slot]
      const float4* sc = reinterpret_cast<const float4*>(s.score + (size_t)blk * hkv * kPage);
      const int n4 = hkv * (kPage / 4);
      for (int i = 0; i < n4; ++i) {
        const float4 v = sc[i];
        acc += (double)v.x;
        acc += (double)v.y;
        acc += (double)v.z;
        acc += (double)v.w;
      }
    } else {
      atomicOr(&s.counters[kCtrStatus], kDevBadBlockId);
    }
    krow[p] = (unsigned long long)__double_as_longlong(acc);
  }
}

template <bool kRelease>
__global__ void __launch_bounds__(kEvictThreads) block_evict_kernel(DevState s, int seq_begin, int recent,
                                                                    double retention,
                                                                    const unsigned long long* __restrict__ keys,
                                                                    uint8_t* __restrict__ mask, int s_cap) {
  __shared__ __align__(16) unsigned long long buf[kMaxBlockPages];  // the keys, then (release) the old row
  __shared__ uint8_t gone[kMaxBlockPages];
  __shared__ int hist[256];
  __shared__ int sh_warp[32];
  __shared__ int sh_sel[3];
  const int bl = blockIdx.x;
  const int b = seq_begin + bl;
  const int S = s.seq_slots[b];
  const int hkv = s.hkv;
  const int n_cand = max(0, S - recent) / kPage;
  const int n_evict = (int)((double)n_cand * (1.0 - retention));
  const int np = S - kPage * n_evict;
  if (threadIdx.x == 0) {
    s.plan[2 * b] = S;
    s.plan[2 * b + 1] = np;
  }
  if (kRelease && n_evict == 0) return;
  const unsigned long long* krow = keys + (size_t)bl * s.max_bps;
  for (int p = threadIdx.x; p < n_cand; p += kEvictThreads) buf[p] = krow[p];
  __syncthreads();

  // ---- the n_evict-th smallest key on the selected bits (prefix / pmask);
  // rem = how many of the keys equal to it there go
  unsigned long long prefix = 0, pmask = 0;
  int rem = n_evict;
  if (n_evict > 0) {
#pragma unroll 1
    for (int pass = 0; pass < 8; ++pass) {
      const int shift = 56 - 8 * pass;
      if (threadIdx.x < 256) hist[threadIdx.x] = 0;
      __syncthreads();
      // lanes of a warp that fall in the same bin add once (the high bytes,
      // mostly the sums' exponents, put most pages in a few bins)
      for (int p0 = 0; p0 < n_cand; p0 += kEvictThreads) {
        const int p = p0 + (int)threadIdx.x;
        const unsigned long long k = p < n_cand ? buf[p] : 0ull;
        const bool on = p < n_cand && (k & pmask) == prefix;
        const int bin = on ? (int)((k >> shift) & 0xFF) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, bin);
        if (on && (threadIdx.x & 31) == (unsigned)(__ffs(peers) - 1)) atomicAdd(&hist[bin], __popc(peers));
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int c[8], sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = hist[8 * lane + j];
          sum += c[j];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int excl = incl - sum;
        if (excl < rem && incl >= rem) {
          int run = excl;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (run + c[j] >= rem) {
              sh_sel[0] = 8 * lane + j;
              sh_sel[1] = rem - run;
              sh_sel[2] = c[j];
              break;
            }
            run += c[j];
          }
        }
      }
      __syncthreads();
      prefix |= (unsigned long long)sh_sel[0] << shift;
      pmask |= 0xFFull << shift;
      rem = sh_sel[1];
      const bool all_of_bin = sh_sel[2] == rem;
      __syncthreads();
      if (all_of_bin) break;  // every key on this prefix goes: the lower bits decide nothing
    }
  }
  // ---- per page: gone = below the prefix, or on it and among the first rem
  // in page order
  int eq_base = 0;
  const int npages = (S + kPage - 1) / kPage;
  for (int c0 = 0; c0 < npages; c0 += kEvictThreads) {
    const int p = c0 + (int)threadIdx.x;
    const bool cand = n_evict > 0 && p < n_cand;
    const unsigned long long km = cand ? (buf[p] & pmask) : 0;
    const bool on = cand && km == prefix;
    int tot;
    const int incl = block_scan<kEvictThreads>(on ? 1 : 0, sh_warp, &tot);
    if (p < npages) gone[p] = (cand && km < prefix) || (on && eq_base + incl - 1 < rem);
    eq_base += tot;
  }
  __syncthreads();

  if (!kRelease) {
    // keep mask of every head: a slot goes when its page goes
    const bool vec = ((reinterpret_cast<uintptr_t>(mask) | (uintptr_t)s_cap) & 15) == 0;
    for (int i = threadIdx.x; i < hkv * npages; i += kEvictThreads) {
      const int h = i / npages, p = i - h * npages;
      uint8_t* m = mask + ((size_t)bl * hkv + h) * s_cap + (size_t)p * kPage;
      const uint8_t v = gone[p] ? 0 : 1;
      if (vec && (p + 1) * kPage <= S) {
        const uint32_t w4 = v * 0x01010101u;
        *reinterpret_cast<uint4*>(m) = make_uint4(w4, w4, w4, w4);
      } else {
        for (int t = 0; t < kPage && p * kPage + t < S; ++t) m[t] = v;
      }
    }
    return;
  }

  // ---- release: the kept pages in order, the dropped ones to the free stack
  int32_t* row = s.block_table + (size_t)b * s.max_bps;
  int32_t* row_in = reinterpret_cast<int32_t*>(buf);
  for (int p = threadIdx.x; p < npages; p += kEvictThreads) row_in[p] = row[p];
  if (threadIdx.x == 0) {
    int base = -1;
    if (n_evict > 0) {
      base = atomicAdd(&s.counters[kCtrFreeTop], n_evict);
      if (base + n_evict > s.num_blocks) {
        atomicSub(&s.counters[kCtrFreeTop], n_evict);
        atomicOr(&s.counters[kCtrStatus], kDevStackOverflow);
        base = -1;
      }
    }
    sh_sel[0] = base;
  }
  __syncthreads();
  const int fbase = sh_sel[0];
  int kept_base = 0, drop_base = 0;
  for (int c0 = 0; c0 < npages; c0 += kEvictThreads) {
    const int p = c0 + (int)threadIdx.x;
    const bool valid = p < npages;
    const bool drop = valid && gone[p];
    const bool keep = valid && !drop;
    int tot;
    const int incl = block_scan<kEvictThreads>((keep ? 1 : 0) | (drop ? 1 << 16 : 0), sh_warp, &tot);
    if (keep) row[kept_base + (incl & 0xFFFF) - 1] = row_in[p];
    const int d_rank = drop_base + (incl >> 16) - 1;
    if (drop && fbase >= 0 && d_rank < n_evict) s.free_stack[fbase + d_rank] = row_in[p];
    kept_base += tot & 0xFFFF;
    drop_base += tot >> 16;
  }
  if (threadIdx.x == 0) {
    if (drop_base != n_evict) atomicOr(&s.counters[kCtrStatus], kDevBadKeepMask);
    if (n_evict > 0) s.seq_slots[b] = np;
  }
}

// The block-table rewrite of a block-granular eviction's keep mask (one CTA
// per sequence): the pages whose slots the mask drops (head 0's row; every
// head's is the same) leave the row, the others keep their order, the dropped
// pages go to the free stack and the sequence holds S - 16 * dropped slots.
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

// Release whole sequences (one CTA each): every page of the row back to the
// free stack, lengths to 0.
__global__ void __launch_bounds__(kBlockThreads) release_seq_kernel(DevState s, int seq_begin) {
  __shared__ int sh_base;
  const int b = seq_begin + blockIdx.x;
  const int S = s.seq_slots[b];
  const int np = (S + kPage - 1) / kPage;
  if (threadIdx.x == 0) {
    int base = -1;
    if (np > 0) {
      base = atomicAdd(&s.counters[kCtrFreeTop], np);
      if (base + np > s.num_blocks) {
        atomicSub(&s.counters[kCtrFreeTop], np);
        atomicOr(&s.counters[kCtrStatus], kDevStackOverflow);
        base = -1;
      }
    }
    sh_base = base;
  }
  __syncthreads();
  const int32_t* row = s.block_table + (size_t)b * s.max_bps;
  if (sh_base >= 0)
    for (int j = threadIdx.x; j < np; j += blockDim.x) s.free_stack[sh_base + j] = row[j];
  if (threadIdx.x == 0) {
    s.seq_slots[b] = 0;
    s.seq_pos[b] = 0;
  }
}

}  // namespace

cudaError_t launch_release_sequences(const DevState& s, int seq_begin, int batch, cudaStream_t st) {
  release_seq_kernel<<<batch, kBlockThreads, 0, st>>>(s, seq_begin);
  return cudaGetLastError();
}

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

cudaError_t launch_block_keys(const DevState& s, int seq_begin, int batch, int recent, int max_cand,
                              unsigned long long* keys, cudaStream_t st) {
  // one thread per candidate page of the longest sequence, in small CTAs so
  // the fp64 chains spread over every SM (any grid is correct: grid-stride)
  const int gx = std::max(1, (max_cand + kKeyThreads - 1) / kKeyThreads);
  dim3 grid(gx, batch);
  block_key_kernel<<<grid, kKeyThreads, 0, st>>>(s, seq_begin, recent, keys);
  return cudaGetLastError();
}

cudaError_t launch_select_blocks(const DevState& s, int seq_begin, int batch, int recent, double retention,
                                 const unsigned long long* keys, uint8_t* keep_mask, int s_cap, cudaStream_t st) {
  block_evict_kernel<false><<<batch, kEvictThreads, 0, st>>>(s, seq_begin, recent, retention, keys, keep_mask, s_cap);
  return cudaGetLastError();
}

cudaError_t launch_evict_blocks(const DevState& s, int seq_begin, int batch, int recent, double retention,
                                const unsigned long long* keys, cudaStream_t st) {
  block_evict_kernel<true><<<batch, kEvictThreads, 0, st>>>(s, seq_begin, recent, retention, keys, nullptr, 0);
  return cudaGetLastError();
}

cudaError_t launch_release_blocks(const DevState& s, int seq_begin, int batch, const uint8_t* keep_mask,
                                  int s_cap, cudaStream_t st) {
  block_release_kernel<<<batch, kBlockThreads, 0, st>>>(s, seq_begin, keep_mask, s_cap);
  return cudaGetLastError();
}

}  // namespace kvc
