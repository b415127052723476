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
#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kCompactThreads = 512;
constexpr int kSelBtStage = 2048;  // block-table entries staged in shared memory

__device__ __forceinline__ size_t slot_index(const DevState& s, const int32_t* bt, int h, int t, bool& ok) {
  const int blk = bt[t / kPage];
  ok = (unsigned)blk < (unsigned)s.num_blocks;
  return ((size_t)(ok ? blk : 0) * s.hkv + h) * kPage + (t % kPage);
}

// Block-wide inclusive sum of one int per thread; returns the thread's
// inclusive prefix and writes the block total to *total.  All threads call it.
template <int NT>
__device__ int block_scan(int v, int* sh_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < NT / 32 ? sh_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < NT / 32) sh_warp[lane] = w;  // inclusive warp prefix
  }
  __syncthreads();
  const int before = warp > 0 ? sh_warp[warp - 1] : 0;
  *total = sh_warp[NT / 32 - 1];
  __syncthreads();
  return before + x;
}

// Radix select over `n` entries: among the entries with active(i) true, find
// the `want`-th in the requested order (largest-first when `descending`) of
// value(i); returns the value and, in *remaining, how many entries equal to it
// are still wanted (1 <= *remaining).
template <typename ActiveF, typename ValueF>
__device__ uint32_t radix_select(int n, int want, bool descending, ActiveF active, ValueF value,
                                 int* hist, int* sh_sel, int* remaining) {
  uint32_t prefix = 0, pmask = 0;
  int rem = want;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      if (!active(i)) continue;
      const uint32_t v = value(i);
      if ((v & pmask) == prefix) atomicAdd(&hist[(v >> shift) & 0xFF], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // warp 0: scan the 256 bins in the requested order, 8 bins per lane
      const int lane = threadIdx.x;
      int cnt[8];
      int sum = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int bin = descending ? 255 - (lane * 8 + k) : lane * 8 + k;
        cnt[k] = hist[bin];
        sum += cnt[k];
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
        for (int k = 0; k < 8; ++k) {
          if (run + cnt[k] >= rem) {
            const int bin = descending ? 255 - (lane * 8 + k) : lane * 8 + k;
            sh_sel[0] = bin;
            sh_sel[1] = rem - run;
            break;
          }
          run += cnt[k];
        }
      }
    }
    __syncthreads();
    prefix |= (uint32_t)sh_sel[0] << shift;
    pmask |= 0xFFu << shift;
    rem = sh_sel[1];
    __syncthreads();
  }
  *remaining = rem;
  return prefix;
}

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
  __shared__ int hist[256];
  __shared__ int sh_sel[2];
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

  int need;
  const uint32_t theta = radix_select(
      S, n_keep, true, [&](int) { return true; }, [&](int i) { return keys[i]; }, hist, sh_sel, &need);
  // ties at theta: how many are there?
  int my_ties = 0;
  for (int t = threadIdx.x; t < S; t += blockDim.x) my_ties += keys[t] == theta;
  int ties;
  block_scan<kSelThreads>(my_ties, sh_warp, &ties);
  uint32_t pos_cut = 0xFFFFFFFFu;
  if (ties > need) {
    int rem2;
    pos_cut = radix_select(
        S, need, false, [&](int i) { return keys[i] == theta; }, [&](int i) { return (uint32_t)pos[i]; }, hist,
        sh_sel, &rem2);
  }
  for (int t = threadIdx.x; t < S; t += blockDim.x) {
    const uint32_t k = keys[t];
    mrow[t] = (k > theta || (k == theta && (uint32_t)pos[t] <= pos_cut)) ? 1 : 0;
  }
}

// Compaction of one (KV head, sequence).  Phase 1 (tiles of 16 slots per
// thread): the keep-mask bytes of a thread's 16 slots come in one 16-byte
// load; block scans give every hole (evicted slot below n') and every source
// (kept slot at or above n') its rank, and the physical pool index of the
// i-th hole and of the i-th source go to two lists.  Phase 2: each warp moves
// several (source -> hole) rows at once, lanes splitting a row 4 bytes each,
// all loads of a batch issued before its stores.
__global__ void __launch_bounds__(kCompactThreads) compact_kernel(DevState s, int seq_begin,
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

  int hole_base = 0, src_base = 0, kept_total = 0;
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
    // bit i of `below` is set when slot t0 + i < n'
    const int nb = min(max(np - t0, 0), 16);
    const uint32_t below = nb >= 16 ? 0xFFFFu : ((1u << nb) - 1u);
    const int nv = min(max(S - t0, 0), 16);
    const uint32_t valid = nv >= 16 ? 0xFFFFu : ((1u << nv) - 1u);
    const uint32_t hole_bits = ~kept_bits & below & valid;
    const uint32_t src_bits = kept_bits & ~below;
    const int nh = __popc(hole_bits), ns = __popc(src_bits), nk = __popc(kept_bits);
    int tot_h, tot_s, tot_k;
    int ph = hole_base + block_scan<kCompactThreads>(nh, sh_warp, &tot_h) - nh;
    int ps = src_base + block_scan<kCompactThreads>(ns, sh_warp, &tot_s) - ns;
    block_scan<kCompactThreads>(nk, sh_warp, &tot_k);
    for (uint32_t m = hole_bits; m; m &= m - 1) {
      const int t = t0 + __ffs(m) - 1;
      holes[ph++] = (bt[t / kPage] * hkv + h) * kPage + (t % kPage);
    }
    for (uint32_t m = src_bits; m; m &= m - 1) {
      const int t = t0 + __ffs(m) - 1;
      srcs[ps++] = (bt[t / kPage] * hkv + h) * kPage + (t % kPage);
    }
    hole_base += tot_h;
    src_base += tot_s;
    kept_total += tot_k;
  }
  if (kept_total != np || hole_base != src_base) {
    if (threadIdx.x == 0) atomicOr(&s.counters[kCtrStatus], kDevBadKeepMask);
    return;
  }
  __syncthreads();

  // phase 2: moves.  A row of codes is row_bytes / 4 words; lanes split it.
  const int n_moves = hole_base;
  const int words = s.row_bytes / 4;            // 32 (INT8) or 16 (INT4)
  const int per_pass = 32 / words;              // moves covered by one warp instruction
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane / words, wl = lane % words;
  constexpr int U = 8;
  const int nwarps = kCompactThreads / 32;
  const uint32_t nslots = (uint32_t)s.num_blocks * hkv * kPage;
  const uint32_t* kc = reinterpret_cast<const uint32_t*>(s.k_codes);
  const uint32_t* vc = reinterpret_cast<const uint32_t*>(s.v_codes);
  for (int base = warp * per_pass * U; base < n_moves; base += nwarps * per_pass * U) {
    uint32_t kw[U], vw[U], si[U], di[U];
    float sc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int mi = base + u * per_pass + sub;
      si[u] = mi < n_moves ? (uint32_t)srcs[mi] : 0xFFFFFFFFu;
      di[u] = mi < n_moves ? (uint32_t)holes[mi] : 0xFFFFFFFFu;
      const bool ok = si[u] < nslots && di[u] < nslots;
      if (!ok) si[u] = di[u] = 0xFFFFFFFFu;
      kw[u] = ok ? kc[(size_t)si[u] * words + wl] : 0u;
      vw[u] = ok ? vc[(size_t)si[u] * words + wl] : 0u;
      sc[u] = 0.0f;
      if (ok && wl < 4) {
        const uint32_t* scal = wl == 0 ? reinterpret_cast<const uint32_t*>(s.k_scale)
                             : wl == 1 ? reinterpret_cast<const uint32_t*>(s.v_scale)
                             : wl == 2 ? reinterpret_cast<const uint32_t*>(s.slot_pos)
                                       : reinterpret_cast<const uint32_t*>(s.score);
        sc[u] = __uint_as_float(scal[si[u]]);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (di[u] == 0xFFFFFFFFu) continue;
      reinterpret_cast<uint32_t*>(s.k_codes)[(size_t)di[u] * words + wl] = kw[u];
      reinterpret_cast<uint32_t*>(s.v_codes)[(size_t)di[u] * words + wl] = vw[u];
      if (wl < 4) {
        uint32_t* scal = wl == 0 ? reinterpret_cast<uint32_t*>(s.k_scale)
                       : wl == 1 ? reinterpret_cast<uint32_t*>(s.v_scale)
                       : wl == 2 ? reinterpret_cast<uint32_t*>(s.slot_pos)
                                 : reinterpret_cast<uint32_t*>(s.score);
        scal[di[u]] = __float_as_uint(sc[u]);
      }
    }
  }
  // release the emptied pages (all KV heads share the page structure)
  if (h == 0) {
    const int keep_pages = (np + kPage - 1) / kPage;
    const int old_pages = (S + kPage - 1) / kPage;
    const int nfree = old_pages - keep_pages;
    __shared__ int sh_base;
    if (threadIdx.x == 0) {
      int base = 0;
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
      for (int i = threadIdx.x; i < nfree; i += blockDim.x) s.free_stack[sh_base + i] = bt[keep_pages + i];
  }
}

}  // namespace

int select_max_smem_slots() { return (200 * 1024) / 8; }

cudaError_t launch_select(const DevState& s, int seq_begin, int batch, const SelectArgs& a, uint8_t* keep_mask,
                          cudaStream_t st) {
  const int smem = a.smem_slots > 0 ? a.smem_slots * 8 : 0;
  if (smem > 48 * 1024) {
    // raise the kernel's dynamic shared-memory limit once per device
    static int done[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64 || !done[dev]) {
      e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               select_max_smem_slots() * 8);
      if (e != cudaSuccess) return e;
      if (dev < 64) done[dev] = 1;
    }
  }
  dim3 grid(s.hkv, batch);
  select_kernel<<<grid, kSelThreads, smem, st>>>(s, seq_begin, a, keep_mask);
  return cudaGetLastError();
}

int compact_max_smem_moves() { return (96 * 1024) / 8; }

cudaError_t launch_compact(const DevState& s, int seq_begin, int batch, const uint8_t* keep_mask, int s_cap,
                           int32_t* g_holes, int32_t* g_srcs, int smem_moves, cudaStream_t st) {
  const int smem = smem_moves > 0 ? smem_moves * 8 : 0;
  if (smem > 48 * 1024) {
    static int done[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64 || !done[dev]) {
      e = cudaFuncSetAttribute(compact_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               compact_max_smem_moves() * 8);
      if (e != cudaSuccess) return e;
      if (dev < 64) done[dev] = 1;
    }
  }
  dim3 grid(s.hkv, batch);
  compact_kernel<<<grid, kCompactThreads, smem, st>>>(s, seq_begin, keep_mask, s_cap, g_holes, g_srcs, smem_moves);
  return cudaGetLastError();
}

}  // namespace kvc
