// Device helpers shared by the kernels of the compressed-KV library: the
// exp2 and bf16 primitives, the page prefix of a batch slice and the stream-K
// CTA lookup of the split attention, block scans and the radix select of the
// kept-set selection, the merge of the split-K partials with the sinks, and
// the compaction's row moves.
#pragma once

#include <cuda_bf16.h>

#include "kvc_internal.h"

namespace kvc {
namespace dev {

constexpr float kNegBig = -1.0e30f;

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16f(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// Pages per sequence of the slice, as an exclusive prefix in shared memory:
// cum[i] = pages of local sequences 0..i-1 (each KV head of a sequence has the
// same pages).  Warp 0 computes it; every thread returns after the barrier.
__device__ __forceinline__ void pages_prefix(const DevState& s, int seq_begin, int batch, int* cum) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    if (lane == 0) cum[0] = 0;
    for (int base = 0; base < batch; base += 32) {
      const int i = base + lane;
      int v = i < batch ? (s.seq_slots[seq_begin + i] + kPage - 1) / kPage : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      if (i < batch) cum[i + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();
}

// CTA of the stream-K split that holds flattened page F (see AttnWork).
__device__ __forceinline__ int cta_of_page(long long F, long long T, int N) {
  return (int)(((F + 1) * (long long)N - 1) / T);
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
// are still wanted (1 <= *remaining) and, in *ties, how many active entries
// equal it.  MSB-first in three passes of 11, 11 and 10 bits: wide digits
// spread values that share their top bits (scores of one magnitude share
// sign and exponent) over many histogram bins, so the shared-memory atomics
// seldom meet on one address.  `hist` holds kRadixBins ints; with
// pass0_ready it already holds the first pass's histogram (bits 31..21 of
// every active value), built by the caller.  The NT threads scan the bins,
// each owning nb / NT consecutive ones in the requested order.  sh_sel holds
// three ints.
constexpr int kRadixBins = 2048;

template <int NT, typename ActiveF, typename ValueF>
__device__ uint32_t radix_select(int n, int want, bool descending, ActiveF active, ValueF value, int* hist,
                                 int* sh_warp, int* sh_sel, int* remaining, int* ties, bool pass0_ready = false) {
  static_assert(NT >= 32 && NT <= 1024 && (1024 % NT) == 0, "block size");
  uint32_t prefix = 0, pmask = 0;
  int rem = want, equal = 0;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass == 2 ? 1024 : kRadixBins;
    if (pass > 0 || !pass0_ready) {
      for (int i = threadIdx.x; i < nb; i += NT) hist[i] = 0;
      __syncthreads();
      for (int i = threadIdx.x; i < n; i += NT) {
        if (!active(i)) continue;
        const uint32_t v = value(i);
        if ((v & pmask) == prefix) atomicAdd(&hist[(v >> shift) & (nb - 1)], 1);
      }
    }
    __syncthreads();
    constexpr int kMaxPer = kRadixBins / NT;
    const int per = nb / NT;
    int cnt[kMaxPer];
    int sum = 0;
#pragma unroll
    for (int k = 0; k < kMaxPer; ++k) {
      cnt[k] = 0;
      if (k < per) {
        const int j = (int)threadIdx.x * per + k;
        cnt[k] = hist[descending ? nb - 1 - j : j];
        sum += cnt[k];
      }
    }
    int total;
    const int incl = block_scan<NT>(sum, sh_warp, &total);
    const int excl = incl - sum;
    if (excl < rem && incl >= rem) {
      int run = excl;
#pragma unroll
      for (int k = 0; k < kMaxPer; ++k) {
        if (k < per && run + cnt[k] >= rem) {
          const int j = (int)threadIdx.x * per + k;
          sh_sel[0] = descending ? nb - 1 - j : j;
          sh_sel[1] = rem - run;
          sh_sel[2] = cnt[k];  // entries matching the prefix so far
          break;
        }
        run += cnt[k];
      }
    }
    __syncthreads();
    prefix |= (uint32_t)sh_sel[0] << shift;
    pmask |= (uint32_t)(nb - 1) << shift;
    rem = sh_sel[1];
    equal = sh_sel[2];
    __syncthreads();
  }
  *remaining = rem;
  *ties = equal;  // after the last pass: the entries equal to the result
  return prefix;
}

// Compaction target: the kept slots of a (sequence, KV head) with S slots
// and n' < S kept end up in the window [w, w + n'), w = the start of the
// last page-aligned window of n' slots inside [0, S).  Evicted slots inside
// the window are the holes, kept slots outside it the sources; afterwards
// the block-table row drops its first w / 16 pages, so the window becomes
// slots [0, n').  After a long prefill the always-kept recent tokens sit at
// the end of the sequence, inside the window, and stay where they are; at
// steady state (S = n' + 1) w = 0.  A function of (S, n') only, so every KV
// head of a sequence uses the same window.
__device__ __forceinline__ int keep_window(int S, int np) { return np < S ? ((S - np) / kPage) * kPage : 0; }

// row[i] = row[p0 + i] for i < n, in place, by the whole block (reads of a
// chunk before its writes; later chunks read only entries past this chunk).
// Starts and ends with a barrier.
__device__ __forceinline__ void shift_row(int32_t* row, int p0, int n) {
  for (int c0 = 0; c0 < n; c0 += blockDim.x) {
    const int i = c0 + (int)threadIdx.x;
    __syncthreads();
    const int32_t v = i < n ? row[p0 + i] : 0;
    __syncthreads();
    if (i < n) row[i] = v;
  }
  __syncthreads();
}

// Shared state of the merge phase.
struct MergeShared {
  float sl[kMaxGroup][kSinks];  // sink logits (log2 domain)
  float M[kMaxGroup];           // global max per query head
  float invL[kMaxGroup];        // 1 / global sum per query head
};

// Merge, for one (sequence bl, KV head h), the stream-K partials of its pages,
// the partials of its bf16 window (hybrid precision, one per chunk that holds
// tokens) and its bf16 sinks: global (M, L) per query head of the group, bf16
// output o = (sum of rescaled partials + sinks) / L, and, with `accumulate`,
// the sink scores' H2O increments.  `cum` is the page prefix of the slice.
// Any block size that is a multiple of 32; ends after a barrier with ms
// filled.
__device__ __forceinline__ void merge_phase(const DevState& s, int seq_begin, int batch, const int* cum, int h,
                                            int bl, const uint16_t* __restrict__ q, uint16_t* __restrict__ out,
                                            float qk_scale_log2, const AttnWork& w, bool accumulate,
                                            MergeShared& ms) {
  const int b = seq_begin + bl;
  const int G = s.group;
  const int hkv = s.hkv;
  const int P = s.seq_pos[b];
  const int ns = min(P, kSinks);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int pair = bl * hkv + h;
  const int npg = cum[bl + 1] - cum[bl];
  const int nrc = (ring_count(P, s.ring) + kRingChunk - 1) / kRingChunk;  // window chunks with tokens
  const float* rpo = w.ring_po + (size_t)pair * w.ring_chunks * G * kHeadDim;
  const float* rpml = w.ring_pml + (size_t)pair * w.ring_chunks * G * 2;
  int i_first = 0, i_last = -1;
  if (npg > 0) {
    const long long T = (long long)hkv * cum[batch];
    const long long Pf = (long long)hkv * cum[bl] + (long long)h * npg;
    i_first = cta_of_page(Pf, T, w.ncta);
    i_last = cta_of_page(Pf + npg - 1, T, w.ncta);
  }
  const uint16_t* sk = s.sink_k + ((size_t)b * hkv + h) * kSinks * kHeadDim;
  const uint16_t* sv = s.sink_v + ((size_t)b * hkv + h) * kSinks * kHeadDim;
  {
    // Everything the merge reads lies in a few contiguous runs: the pair's
    // partials (consecutive slots pair + i_first .. pair + i_last), its
    // query rows and sink rows.  Prefetch them into L1 now, so the phases
    // after each barrier below find them there instead of in L2.
    const int npart = i_last - i_first + 1;
    const char* po = reinterpret_cast<const char*>(w.part_o + ((size_t)pair + i_first) * G * kHeadDim);
    const char* pm = reinterpret_cast<const char*>(w.part_ml + ((size_t)pair + i_first) * G * 2);
    const char* qr = reinterpret_cast<const char*>(q + ((size_t)bl * s.hq + h * G) * kHeadDim);
    const int lo = npart * G * kHeadDim * 4 / 128;             // part_o lines
    const int lm = (npart * G * 2 * 4 + 127) / 128;            // part_ml lines
    const int lq = G * kHeadDim * 2 / 128;                     // query lines
    const int ls = kSinks * kHeadDim * 2 / 128;                // lines per sink tensor
    for (int i = threadIdx.x; i < lo + lm + lq + 2 * ls; i += blockDim.x) {
      const char* a = i < lo ? po + 128 * i
                    : i < lo + lm ? pm + 128 * (i - lo)
                    : i < lo + lm + lq ? qr + 128 * (i - lo - lm)
                    : i < lo + lm + lq + ls ? reinterpret_cast<const char*>(sk) + 128 * (i - lo - lm - lq)
                                            : reinterpret_cast<const char*>(sv) + 128 * (i - lo - lm - lq - ls);
      asm volatile("prefetch.global.L1 [%0];" ::"l"(a));
    }
  }

  // sink logits: warp task (g, j) = (task / 4, task % 4)
  for (int task = warp; task < kMaxGroup * kSinks; task += nwarps) {
    const int g = task >> 2, j = task & 3;
    if (g < G) {
      float part = 0.0f;
      if (j < ns) {
        const uint16_t* qr = q + ((size_t)bl * s.hq + h * G + g) * kHeadDim;
#pragma unroll
        for (int e = 0; e < 4; ++e) part += bf16f(qr[lane * 4 + e]) * bf16f(sk[j * kHeadDim + lane * 4 + e]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if (lane == 0) ms.sl[g][j] = j < ns ? part * qk_scale_log2 : -INFINITY;
    }
  }
  __syncthreads();
  // global max and sum per query head: warp g
  if (warp < G) {
    const int g = warp;
    float M = kNegBig;
    for (int i = i_first + lane; i <= i_last; i += 32) M = fmaxf(M, w.part_ml[(((size_t)pair + i) * G + g) * 2]);
    for (int i = lane; i < nrc; i += 32) M = fmaxf(M, rpml[((size_t)i * G + g) * 2]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
#pragma unroll
    for (int j = 0; j < kSinks; ++j) M = fmaxf(M, ms.sl[g][j]);
    float L = 0.0f;
    for (int i = i_first + lane; i <= i_last; i += 32) {
      const size_t pi = ((size_t)pair + i) * G + g;
      L += fast_exp2(w.part_ml[pi * 2] - M) * w.part_ml[pi * 2 + 1];
    }
    for (int i = lane; i < nrc; i += 32) {
      const size_t pi = (size_t)i * G + g;
      L += fast_exp2(rpml[pi * 2] - M) * rpml[pi * 2 + 1];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < kSinks; ++j)
        if (j < ns) L += fast_exp2(ms.sl[g][j] - M);
      ms.M[g] = M;
      ms.invL[g] = L > 0.0f ? 1.0f / L : 0.0f;
      w.stats[((size_t)bl * s.hq + h * G + g) * 2 + 0] = M;
      w.stats[((size_t)bl * s.hq + h * G + g) * 2 + 1] = L;
    }
  }
  __syncthreads();
  // outputs: thread (g, d)
  for (int gd = threadIdx.x; gd < G * kHeadDim; gd += blockDim.x) {
    const int g = gd >> 7, d = gd & (kHeadDim - 1);
    const float M = ms.M[g];
    float o = 0.0f;
#pragma unroll
    for (int j = 0; j < kSinks; ++j)
      if (j < ns) o += fast_exp2(ms.sl[g][j] - M) * bf16f(sv[j * kHeadDim + d]);
    for (int i = i_first; i <= i_last; ++i) {
      const size_t pi = ((size_t)pair + i) * G + g;
      o += fast_exp2(w.part_ml[pi * 2] - M) * w.part_o[pi * kHeadDim + d];
    }
    for (int i = 0; i < nrc; ++i) {
      const size_t pi = (size_t)i * G + g;
      o += fast_exp2(rpml[pi * 2] - M) * rpo[pi * kHeadDim + d];
    }
    out[((size_t)bl * s.hq + h * G + g) * kHeadDim + d] = __bfloat16_as_ushort(__float2bfloat16_rn(o * ms.invL[g]));
  }
  if (accumulate && (int)threadIdx.x < ns) {
    float inc = 0.0f;
    for (int g = 0; g < G; ++g) inc += fast_exp2(ms.sl[g][threadIdx.x] - ms.M[g]) * ms.invL[g];
    s.sink_score[((size_t)b * hkv + h) * kSinks + threadIdx.x] += inc;
  }
}

// H2O increments of the bf16 window's tokens (hybrid precision), from the
// logits the window attention spilled; same arithmetic and order as
// h2o_increment.  After merge_phase (ms filled); any block size.
__device__ __forceinline__ void ring_score_pass(const DevState& s, const AttnWork& w, int b, int bl, int h,
                                                const MergeShared& ms) {
  const int W = s.ring;
  if (W <= 0) return;
  const int G = s.group;
  const int nr = ring_count(s.seq_pos[b], W);
  const float* lg = w.ring_lg + ((size_t)bl * s.hkv + h) * G * W;
  float* sc = s.ring_score + ((size_t)b * s.hkv + h) * W;
  for (int r = threadIdx.x; r < nr; r += blockDim.x) {
    float inc = 0.0f;
    for (int g = 0; g < G; ++g) inc = __fmaf_rn(fast_exp2(lg[(size_t)g * W + r] - ms.M[g]), ms.invL[g], inc);
    sc[r] += inc;
  }
}

// Pool slot index of slot t of a sequence's row for KV head h, or -1 (which
// move_rows rejects) when the row's block id is outside the pool.
__device__ __forceinline__ int32_t slot_index(const DevState& s, const int32_t* row, int t, int h) {
  const int blk = row[t / kPage];
  return (unsigned)blk < (unsigned)s.num_blocks ? (blk * s.hkv + h) * kPage + (t % kPage) : -1;
}

// H2O increment of one pool slot: sum over the G query heads of its softmax
// probability, from the spilled log2-domain logits ([g][slot] rows).
__device__ __forceinline__ float h2o_increment(const float* lgr, int s_cap, int t, int G, const MergeShared& ms) {
  float inc = 0.0f;
  for (int g = 0; g < G; ++g) inc = __fmaf_rn(fast_exp2(lgr[(size_t)g * s_cap + t] - ms.M[g]), ms.invL[g], inc);
  return inc;
}

// Row moves of one (KV head, sequence): entry i of `srcs` (a physical pool
// slot) goes to entry i of `holes`, with its K and V code rows, scales,
// position and score.  The row_bytes / 16 lanes of a row move its 16-byte
// chunks in one instruction, so every store covers whole 32-byte sectors (a
// store of half a sector makes L2 fetch the sector from DRAM first); a warp
// moves 32 / (row_bytes / 16) consecutive entries per instruction, three such
// groups in flight.  The lane holding chunk 0 of a row also moves the slot's
// four scalars.  Entries outside the pool set kDevBadBlockId and are skipped.
__device__ __forceinline__ void move_rows(const DevState& s, const int32_t* holes, const int32_t* srcs,
                                          int n_moves) {
  constexpr int U = 3;
  const uint32_t nslots = (uint32_t)s.num_blocks * s.hkv * kPage;
  const int lpr = s.row_bytes / 16;  // lanes per row
  const int rpw = 32 / lpr;          // rows per warp instruction
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int r = lane / lpr, c = lane % lpr;
  const int stride = nwarps * rpw * U;
  // the list entries of the next round are loaded while this round's rows
  // are in flight (one memory round trip per round instead of two)
  uint32_t nsi[U], ndi[U];
  auto load_lists = [&](int base) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int mi = base + u * rpw + r;
      nsi[u] = mi < n_moves ? (uint32_t)srcs[mi] : 0xFFFFFFFFu;
      ndi[u] = mi < n_moves ? (uint32_t)holes[mi] : 0xFFFFFFFFu;
    }
  };
  load_lists(warp * rpw * U);
  for (int base = warp * rpw * U; base < n_moves; base += stride) {
    uint4 kv[U], vv[U];
    uint32_t si[U], di[U];
    bool on[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int mi = base + u * rpw + r;
      on[u] = mi < n_moves;
      si[u] = nsi[u];
      di[u] = ndi[u];
      if (on[u] && (si[u] >= nslots || di[u] >= nslots)) {
        if (c == 0) atomicOr(&s.counters[kCtrStatus], kDevBadBlockId);
        on[u] = false;
      }
      if (on[u]) {
        kv[u] = reinterpret_cast<const uint4*>(s.k_codes + (size_t)si[u] * s.row_bytes)[c];
        vv[u] = reinterpret_cast<const uint4*>(s.v_codes + (size_t)si[u] * s.row_bytes)[c];
      }
    }
    float ks[U], vs[U], sc[U];
    int ps[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (on[u] && c == 0) {
        ks[u] = s.k_scale[si[u]];
        vs[u] = s.v_scale[si[u]];
        sc[u] = s.score[si[u]];
        ps[u] = s.slot_pos[si[u]];
      }
    }
    load_lists(base + stride);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!on[u]) continue;
      reinterpret_cast<uint4*>(s.k_codes + (size_t)di[u] * s.row_bytes)[c] = kv[u];
      reinterpret_cast<uint4*>(s.v_codes + (size_t)di[u] * s.row_bytes)[c] = vv[u];
      if (c == 0) {
        s.k_scale[di[u]] = ks[u];
        s.v_scale[di[u]] = vs[u];
        s.score[di[u]] = sc[u];
        s.slot_pos[di[u]] = ps[u];
      }
    }
  }
}

}  // namespace dev
}  // namespace kvc
