// A prompt over sequences that already hold context (a later turn): every
// prompt query attends, as a decode step would, to the tokens the compressed
// cache holds at positions up to its own, and adds its probabilities to their
// H2O scores (the eviction-and-reuse survey page, section 3.3: a token's
// score is its cumulative attention from the later tokens; the Technical
// Report, section 3.4: the column sums of the attention matrix; the
// dequantisation fused into the attention, section 3.2).
//
// After the prompt's append, the keys of one (sequence, KV head) are the
// sinks followed by the pool slots in slot order, and the prompt's own pool
// tokens are the last slots, in position order.  So what prompt query i
// (position P0 + i) may see is the sinks at positions <= P0 + i and a prefix
// of the pool: vis(i) = S0 + max(0, P0 + i + 1 - max(P0, 4)) slots, S0 the
// slots before the prompt.  That is a causal mask shifted by the context.
//
// GB300 design: the rows of the attention matrix of one (sequence, KV head)
// are its prompt queries times the G query heads of the group (row = i G + g);
// a warp owns 16 rows (one MMA row tile) and a CTA of 4 warps streams the
// pool pages its rows may see once through shared memory (cp.async, a
// conflict-free chunk permutation), every warp reading every page:
//   S = Q K^T   mma.sync m16n8k16, the query rows on M (A operand in
//               registers), the page's 16 tokens on N, the codes entering as
//               offset fp16 subnormals exactly as in the decode kernel;
//   O += P V    P straight from the S accumulators (their layout is the A
//               operand's), V on N per 8 head dims.
// Two passes over the pages, so that the column sums use the final
// probabilities: pass 0 finds every row's softmax maximum and sum (sinks
// included); pass 1 recomputes S with the same instructions (the same
// logits), forms p = 2^(s - M) / L, accumulates O and, per page token, the
// sum of p over the CTA's rows into a per-CTA row of column sums.  The last
// CTA of each (sequence, KV head) to finish (an atomic ticket; no CTA waits)
// adds those rows, in CTA order, to the tokens' scores: deterministic.
#include <cuda_bf16.h>

#include <type_traits>

#include "kvc_device.h"
#include "kvc_internal.h"
#include "kvc_mma.h"

namespace kvc {
namespace {

using namespace dev;
using namespace codes;

constexpr int kCtxWarps = 4;
constexpr int kCtxThreads = kCtxWarps * 32;
constexpr int kCtxStages = 4;  // pages in flight per CTA
constexpr float kCtxLazy = 4.0f;

// One stage: the 16 K rows and 16 V rows of a page of one head, its 16 K and
// 16 V scales.  The 16-byte chunks of the code rows are permuted so that the
// copies and the reads of this kernel touch every shared-memory bank at most
// once per 128 bytes: chunk j of row t goes to
//   INT4 (4 chunks a row): 128 (t >> 1) + 16 (4 ((t ^ t >> 1) & 1) + ((j + 2 ((t >> 2) & 1)) & 3)),
//   8-bit (8 chunks a row): 128 t + 16 (j ^ 2 ((t >> 1) & 3) ^ 4 (t & 1)).
template <int BITS>
struct CtxGeom {
  static constexpr int kRowBytes = BITS * 16;
  static constexpr int kK = 0;
  static constexpr int kV = 16 * kRowBytes;
  static constexpr int kKS = 32 * kRowBytes;
  static constexpr int kVS = kKS + 64;
  static constexpr int kStage = kVS + 64;
  static constexpr int kChunksPerRow = kRowBytes / 16;
  static __host__ __device__ constexpr int chunk_off(int t, int j) {
    return BITS == 4 ? 128 * (t >> 1) + 16 * (4 * (((t >> 1) ^ t) & 1) + ((j + 2 * ((t >> 2) & 1)) & 3))
                     : 128 * t + 16 * (j ^ (2 * ((t >> 1) & 3)) ^ (4 * (t & 1)));
  }
};

struct CtxArgs {
  const uint16_t* q;  // [batch][hq][n][128]
  uint16_t* out;      // [batch][hq][n][128]
  float* stats;       // [pairs][rows][2]  (max in the log2 domain, sum)
  float* colsum;      // [pairs][groups][4 + s_cap]  per-CTA column sums (sinks first)
  int* ticket;        // [pairs]
  int n, groups, s_cap;
  int cs_row;         // 4 + s_cap + W: sinks, pool slots, window positions from rlo
  float qk_scale_log2;
  int accumulate;
};

// Lengths of sequence b after the prompt's append: the positions before it
// (P0) and now (P1), the pool slots now (S1).  The append moved positions
// [a, rlo) into the pool, in position order, after the S0 slots it held
// (a = max(4, P0 - W): with a bf16 window of W positions these are the
// window's tokens that aged out and the prompt's own tokens that did; without
// one, the prompt's non-sink tokens); the window holds [rlo, P1).
struct CtxLens {
  int S0, P0, S1, P1, a, rlo;
};
__device__ __forceinline__ CtxLens ctx_lens(const DevState& s, int b, int n) {
  CtxLens l;
  l.S1 = s.seq_slots[b];
  l.P1 = s.seq_pos[b];
  l.P0 = l.P1 - n;
  l.a = max(kSinks, l.P0 - s.ring);
  l.rlo = max(l.a, l.P1 - s.ring);
  l.S0 = l.S1 - (l.rlo - l.a);
  return l;
}
// pool slots query i (position P0 + i) sees: the S0 older ones and the
// appended ones at positions <= P0 + i
__device__ __forceinline__ int ctx_vis(const CtxLens& l, int i) {
  return l.S0 + min(max(l.P0 + i + 1 - l.a, 0), l.rlo - l.a);
}
// window positions query i sees: [rlo, ctx_ring_end)
__device__ __forceinline__ int ctx_ring_end(const CtxLens& l, int i) { return min(l.P1, l.P0 + i + 1); }

// One stage of the window tiles: 16 K rows and 16 V rows of 128 bf16, each
// row padded to 272 bytes (ldmatrix reads them without bank conflicts).
constexpr int kRingRow = 136;  // bf16 per staged row
constexpr int kRingStage = 2 * 16 * kRingRow * 2;

// PASS 0: row statistics; PASS 1: outputs and column sums.
// WIN: the cache keeps a bf16 window (its tiles follow the pool's pages).
// Pass 1 over integer 8-bit codes, and over INT4 codes with a window, is
// held to 168 registers (three CTAs per SM, as the INT4 and FP8 forms
// without a window reach unbounded): it is latency-bound, and unbounded it
// took 239 and 255 registers and ran two CTAs per SM; bounded it spills
// nothing.  Pass 0 over INT4 codes is held to 96 registers (five CTAs per
// SM instead of four, no spills; over 8-bit codes that was slower).  The
// other forms keep the compiler's own choice (a minimum of 0 CTAs per SM
// states none; a minimum of 1 made it spend up to 255 registers on pass 0
// and INT4 pass 1; the 8-bit window forms would spill).
template <int BITS, bool FP8, int PASS, bool WIN>
__global__ void __launch_bounds__(kCtxThreads,
                                  (PASS == 1 && ((BITS == 8 && !FP8 && !WIN) || (BITS == 4 && WIN)))
                                      ? 3
                                      : ((PASS == 0 && BITS == 4) ? 5 : 0))
    ctx_attn_kernel(DevState s, int seq_begin, CtxArgs a) {
  using Gm = CtxGeom<BITS>;
  constexpr int RB = Gm::kRowBytes;
  constexpr int ST = kCtxStages;
  constexpr bool kOffset = !FP8;
  constexpr float kOffK = BITS == 8 ? 128.0f * 0x1p-24f : 8.0f * 0x1p-24f;
  constexpr float kOffV = BITS == 8 ? 128.0f : 8.0f;
  constexpr bool kNeedV = PASS == 1;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float sh_cs[2][kCtxWarps][16];  // pass 1: a page's column sums per warp (by page parity)
  __shared__ float sh_sk[kCtxWarps][kSinks];  // pass 1: the sinks' column sums per warp
  __shared__ int sh_last;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, tq = lane & 3;  // MMA fragment coordinates (group, thread in group)
  const int G = s.group, hkv = s.hkv;
  const int pair = blockIdx.y;
  const int bl = pair / hkv, h = pair % hkv;
  const int b = seq_begin + bl;
  const int mg = blockIdx.x;
  const int n = a.n;
  const int R = n * G;
  const int mtiles = (R + 15) / 16;
  const CtxLens L = ctx_lens(s, b, n);
  const int32_t* bt = s.block_table + (size_t)b * s.max_bps;
  const int n_sinks = min(kSinks, L.P0 + n);
  const uint32_t ring = smem_u32(smem);

  // what this thread copies of a page: K chunk t (and, pass 1, V chunk t) of
  // the 16 * RB / 16 chunks of each run; threads 0..7 one chunk of scales
  constexpr int kChunks = RB;  // 16-byte chunks in a K run
  const bool cp_k = threadIdx.x < kChunks;
  const int ck = threadIdx.x % kChunks;
  const uint32_t cp_dst = Gm::chunk_off(ck / Gm::kChunksPerRow, ck % Gm::kChunksPerRow);
  // pass 0 copies K only: with INT4 (64 chunks) the upper half of the threads
  // have nothing to copy; pass 1 gives them the V run
  const bool cp_v = kNeedV && (BITS == 8 || threadIdx.x >= kChunks);
  const bool cp_kk = BITS == 8 || threadIdx.x < kChunks;
  const uint32_t cp_soff = threadIdx.x < 4 ? Gm::kKS + 16 * threadIdx.x : Gm::kVS + 16 * (threadIdx.x & 3);
  const float* cp_sbase = (threadIdx.x < 4 ? s.k_scale : s.v_scale) + 4 * (threadIdx.x & 3);
  const bool cp_s = threadIdx.x < (kNeedV ? 8 : 4);

  // what this lane reads: K rows g and 8 + g (chunk tq; 8-bit also tq + 4), V
  // rows 2tq, 2tq + 1, 2tq + 8, 2tq + 9 (8 bytes at 8g, or 16 at 16g), the
  // scales of tokens 2tq, 2tq + 1 and 8 + 2tq, 9 + 2tq
  int koff[2][2], voff[4];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    koff[t][0] = Gm::kK + Gm::chunk_off(8 * t + g, tq);
    koff[t][1] = Gm::kK + Gm::chunk_off(8 * t + g, (tq + 4) % Gm::kChunksPerRow);
  }
  {
    const int vr[4] = {2 * tq, 2 * tq + 1, 2 * tq + 8, 2 * tq + 9};
#pragma unroll
    for (int u = 0; u < 4; ++u)
      voff[u] = Gm::kV + (BITS == 8 ? Gm::chunk_off(vr[u], g) : Gm::chunk_off(vr[u], g >> 1) + 8 * (g & 1));
  }

  // block ids of the sequence's pages, staged once (the rounds reuse them)
  const int npages_all = (L.S1 + kPage - 1) / kPage;
  constexpr int kRingBytes = WIN && 2 * kRingStage > ST * Gm::kStage ? 2 * kRingStage : ST * Gm::kStage;
  int32_t* sbt = reinterpret_cast<int32_t*>(smem + kRingBytes);
  const int n_stage_bt = min(npages_all, kCtxBtStage);
  for (int i = threadIdx.x; i < n_stage_bt; i += kCtxThreads) sbt[i] = bt[i];
  if (PASS == 0 && mg == 0 && threadIdx.x == 0) a.ticket[pair] = 0;
  __syncthreads();
  auto blk_of = [&](int p) -> int { return p < kCtxBtStage ? sbt[p] : bt[p]; };

  float* colsum = a.colsum + ((size_t)pair * a.groups + mg) * a.cs_row;
  float* cs_ring = colsum + kSinks + a.s_cap;
  // sink keys and values of this (sequence, KV head)
  const uint16_t* sink_k = s.sink_k + ((size_t)b * hkv + h) * kSinks * kHeadDim;
  const uint16_t* sink_v = s.sink_v + ((size_t)b * hkv + h) * kSinks * kHeadDim;

  // the CTA's rounds: warp w takes row tile mg * 4 + w + 4 * groups * round
  const int rounds = (mtiles + 4 * a.groups - 1) / (4 * a.groups);
  for (int round = 0; round < rounds; ++round) {
    const int tile = (round * a.groups + mg) * kCtxWarps + warp;
    const int row0 = 16 * tile;
    const bool active = row0 < R;
    // the rows of this lane: r_lo = row0 + g, r_hi = row0 + 8 + g
    const int r_lo = row0 + g, r_hi = row0 + 8 + g;
    const bool ok_lo = r_lo < R, ok_hi = r_hi < R;
    const int i_lo = ok_lo ? r_lo / G : 0, i_hi = ok_hi ? r_hi / G : 0;
    const int lim_lo = ok_lo ? ctx_vis(L, i_lo) : 0, lim_hi = ok_hi ? ctx_vis(L, i_hi) : 0;
    // visible slots of the CTA's rows in this round (pages to stream) and of this warp's
    int cta_lim = 0;
    {
      const int last_row = min(R, 16 * ((round * a.groups + mg) * kCtxWarps + kCtxWarps)) - 1;
      if (last_row >= 16 * (round * a.groups + mg) * kCtxWarps) cta_lim = ctx_vis(L, last_row / G);
    }
    const int wfirst = active ? ctx_vis(L, row0 / G) : 0;                       // every row sees these
    const int wlast = active ? ctx_vis(L, (min(R, row0 + 16) - 1) / G) : 0;     // some row sees these
    const int npages = (cta_lim + kPage - 1) / kPage;
    // window tiles (16 positions from rlo) the CTA's rows see, and the window
    // positions this warp's rows see
    int nrt = 0, wring_end = 0;
    if (WIN && s.ring > 0) {
      const int last_row = min(R, 16 * ((round * a.groups + mg) * kCtxWarps + kCtxWarps)) - 1;
      if (last_row >= 16 * (round * a.groups + mg) * kCtxWarps)
        nrt = (max(0, ctx_ring_end(L, last_row / G) - L.rlo) + 15) / 16;
      wring_end = active ? ctx_ring_end(L, (min(R, row0 + 16) - 1) / G) : 0;
      if (PASS == 1 && round == 0)
        for (int e2 = threadIdx.x; e2 < L.P1 - L.rlo; e2 += kCtxThreads) cs_ring[e2] = 0.0f;
    }

    // ---- query fragments (A operand), rows r_lo / r_hi, scaled by 2^e into
    // fp16 range; the offset sum per row; the sink logits per row
    uint32_t qa[8][4];
    float ch_lo = 0.0f, ch_hi = 0.0f, cq_lo = 0.0f, cq_hi = 0.0f;
    float sk_lg[2][kSinks];
    int e_row[2] = {0, 0};
    {
      float qv[2][32];
      float amax[2] = {0.0f, 0.0f};
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int row = rr ? r_hi : r_lo;
        const bool ok = rr ? ok_hi : ok_lo;
        if (ok && active) {
          const int i = row / G, gq = row % G;
          const uint16_t* qrow = a.q + (((size_t)bl * s.hq + h * G + gq) * n + i) * kHeadDim;
          const uint4* src_a = reinterpret_cast<const uint4*>(qrow + (BITS == 8 ? 16 * tq : 32 * tq));
          const uint4* src_b = reinterpret_cast<const uint4*>(qrow + (BITS == 8 ? 64 + 16 * tq : 32 * tq + 16));
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint4 v = u < 2 ? src_a[u] : src_b[u - 2];
            const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              qv[rr][8 * u + 2 * j] = bf16f(ws[j] & 0xFFFFu);
              qv[rr][8 * u + 2 * j + 1] = bf16f(ws[j] >> 16);
            }
          }
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u) qv[rr][u] = 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 32; ++u) amax[rr] = fmaxf(amax[rr], fabsf(qv[rr][u]));
        amax[rr] = fmaxf(amax[rr], __shfl_xor_sync(0xffffffffu, amax[rr], 1));
        amax[rr] = fmaxf(amax[rr], __shfl_xor_sync(0xffffffffu, amax[rr], 2));
      }
      int* e = e_row;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        e[rr] = amax[rr] > 0.0f ? min(max(14 - exponent_of(amax[rr]), -100), 100) : 0;
        // sink logits: q . k_sink over this lane's 32 dims (bf16 products are
        // exact in fp32), summed over the 4 lanes of the row
        const int d0 = BITS == 8 ? 16 * tq : 32 * tq, d1 = BITS == 8 ? 64 + 16 * tq : 32 * tq + 16;
#pragma unroll
        for (int sk = 0; sk < kSinks; ++sk) {
          float acc = 0.0f;
          if (sk < n_sinks) {
            const uint16_t* kr = sink_k + sk * kHeadDim;
#pragma unroll
            for (int u = 0; u < 32; ++u) acc = fmaf(qv[rr][u], bf16f(kr[u < 16 ? d0 + u : d1 + u - 16]), acc);
          }
          acc += __shfl_xor_sync(0xffffffffu, acc, 1);
          acc += __shfl_xor_sync(0xffffffffu, acc, 2);
          sk_lg[rr][sk] = acc * a.qk_scale_log2;
        }
        const float f2e = pow2i(e[rr]);
#pragma unroll
        for (int u = 0; u < 32; ++u) qv[rr][u] *= f2e;
      }
      // A fragments: register 0 row g, register 1 row g + 8 (k-indices 2tq,
      // 2tq+1), registers 2 and 3 the same rows at k-indices 2tq+8, 2tq+9; the
      // dims follow the order of the lane's codes as in the decode kernel
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        if (BITS == 8) {
#pragma unroll
          for (int st = 0; st < 8; ++st) {
            if (FP8) {
              qa[st][rr] = pack_half2(qv[rr][4 * st + 0], qv[rr][4 * st + 1]);
              qa[st][2 + rr] = pack_half2(qv[rr][4 * st + 2], qv[rr][4 * st + 3]);
            } else {
              qa[st][rr] = pack_half2(qv[rr][4 * st + 0], qv[rr][4 * st + 2]);
              qa[st][2 + rr] = pack_half2(qv[rr][4 * st + 1], qv[rr][4 * st + 3]);
            }
          }
        } else {
          constexpr float k16 = 0.0625f;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            qa[2 * m][rr] = pack_half2(qv[rr][8 * m + 0], qv[rr][8 * m + 4]);
            qa[2 * m][2 + rr] = pack_half2(qv[rr][8 * m + 1] * k16, qv[rr][8 * m + 5] * k16);
            qa[2 * m + 1][rr] = pack_half2(qv[rr][8 * m + 2], qv[rr][8 * m + 6]);
            qa[2 * m + 1][2 + rr] = pack_half2(qv[rr][8 * m + 3] * k16, qv[rr][8 * m + 7] * k16);
          }
        }
        float qs = 0.0f;
        if (kOffset) {
#pragma unroll
          for (int st = 0; st < 8; ++st) {
            const float2 x = unpack_half2(qa[st][rr]);
            const float2 y = unpack_half2(qa[st][2 + rr]);
            qs += (x.x + x.y) + (BITS == 4 ? 16.0f : 1.0f) * (y.x + y.y);
          }
          qs += __shfl_xor_sync(0xffffffffu, qs, 1);
          qs += __shfl_xor_sync(0xffffffffu, qs, 2);
        }
        const float cq = a.qk_scale_log2 * pow2i((kOffset ? 24 : 0) - e[rr]);
        if (rr == 0) {
          ch_lo = kOffK * qs;
          cq_lo = cq;
        } else {
          ch_hi = kOffK * qs;
          cq_hi = cq;
        }
      }
    }
    // sinks this row may see: positions <= P0 + i
    const int ns_lo = ok_lo ? min(n_sinks, L.P0 + i_lo + 1) : 0, ns_hi = ok_hi ? min(n_sinks, L.P0 + i_hi + 1) : 0;

    // ---- pass 0: running max and sum per row, starting from the sinks
    float m_lo = kNegBig, m_hi = kNegBig, l_lo = 0.0f, l_hi = 0.0f;
    // ---- pass 1: the final statistics, the output accumulators
    float M_lo = 0.0f, M_hi = 0.0f, iL_lo = 0.0f, iL_hi = 0.0f;
    float oacc[16][4];
    float osum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    int E = 0;
    bool e_set = false;
    float sv_hi = 0.0f, inv2E = 1.0f;
    if (PASS == 0) {
#pragma unroll
      for (int sk = 0; sk < kSinks; ++sk) {
        if (sk < ns_lo) m_lo = fmaxf(m_lo, sk_lg[0][sk]);
        if (sk < ns_hi) m_hi = fmaxf(m_hi, sk_lg[1][sk]);
      }
      if (tq == 0) {  // the sinks count once per row
#pragma unroll
        for (int sk = 0; sk < kSinks; ++sk) {
          if (sk < ns_lo) l_lo += fast_exp2(sk_lg[0][sk] - m_lo);
          if (sk < ns_hi) l_hi += fast_exp2(sk_lg[1][sk] - m_hi);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.0f;
      if (active) {
        const size_t srow = (size_t)pair * R;
        if (ok_lo) {
          const float2 st = *reinterpret_cast<const float2*>(a.stats + (srow + r_lo) * 2);
          M_lo = st.x;
          iL_lo = 1.0f / st.y;
        }
        if (ok_hi) {
          const float2 st = *reinterpret_cast<const float2*>(a.stats + (srow + r_hi) * 2);
          M_hi = st.x;
          iL_hi = 1.0f / st.y;
        }
      }
    }

    // ---- the page stream
    auto issue = [&](int p) {
      if (p < npages) {
        const int blk = blk_of(p);
        const bool okb = (unsigned)blk < (unsigned)s.num_blocks;
        const uint32_t sb = ring + (p % ST) * Gm::kStage;
        const size_t hp = (size_t)(okb ? blk : 0) * hkv + h;
        if (cp_kk) cp_async16_if(okb && cp_k, sb + Gm::kK + cp_dst, s.k_codes + hp * (16 * RB) + 16 * ck);
        if (cp_v) cp_async16_if(okb, sb + Gm::kV + cp_dst, s.v_codes + hp * (16 * RB) + 16 * ck);
        cp_async16_if(okb && cp_s, sb + cp_soff, cp_sbase + hp * kPage);
        if (!okb && threadIdx.x == 0) atomicOr(&s.counters[kCtrStatus], kDevBadBlockId);
      }
      cp_async_commit();
    };
#pragma unroll 1
    for (int p = 0; p < ST - 1; ++p) issue(p);

#pragma unroll 1
    for (int p = 0; p < npages; ++p) {
      cp_async_wait<ST - 2>();
      __syncthreads();  // page p is in; every warp is done with page p - 1
      if (PASS == 1 && p > 0 && threadIdx.x < 16) {
        // the column sums of page p - 1 over the CTA's rows (warps in order)
        const int slot = (p - 1) * kPage + threadIdx.x;
        if (slot < L.S1) {
          const int pb = (p - 1) & 1;
          float v = sh_cs[pb][0][threadIdx.x];
#pragma unroll
          for (int w2 = 1; w2 < kCtxWarps; ++w2) v += sh_cs[pb][w2][threadIdx.x];
          colsum[kSinks + slot] = round == 0 ? v : colsum[kSinks + slot] + v;
        }
      }
      issue(p + ST - 1);
      const int slot0 = p * kPage;
      const bool blk_ok = (unsigned)blk_of(p) < (unsigned)s.num_blocks;
      const bool live = active && blk_ok && slot0 < wlast;
      float cs_t[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // pass 1: this lane's token sums
      if (live) {
        const uint8_t* st = smem + (p % ST) * Gm::kStage;
        const bool full = slot0 + kPage <= wfirst && slot0 + kPage <= L.S1;
        // S = Q K^T: N-tile t = tokens 8t .. 8t+7
        float acc[2][4];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          acc[t][0] = acc[t][1] = -ch_lo;
          acc[t][2] = acc[t][3] = -ch_hi;
        }
        if (BITS == 8) {
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const uint4 x0 = *reinterpret_cast<const uint4*>(st + koff[t][0]);
            const uint4 x1 = *reinterpret_cast<const uint4*>(st + koff[t][1]);
            const uint32_t wv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int stp = 0; stp < 8; ++stp) {
              uint32_t b0, b1;
              if (FP8) {
                e4m3x4_to_h2(wv[stp], b0, b1);
              } else {
                b0 = u8_even(wv[stp]);
                b1 = u8_even(wv[stp] >> 8);
              }
              mma16816(acc[t], qa[stp][0], qa[stp][1], qa[stp][2], qa[stp][3], b0, b1);
            }
          }
        } else {
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const uint4 x = *reinterpret_cast<const uint4*>(st + koff[t][0]);
            const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const uint32_t w0 = wv[m], w1 = wv[m] >> 8;
              mma16816(acc[t], qa[2 * m][0], qa[2 * m][1], qa[2 * m][2], qa[2 * m][3], u4_lo(w0), u4_hi(w0));
              mma16816(acc[t], qa[2 * m + 1][0], qa[2 * m + 1][1], qa[2 * m + 1][2], qa[2 * m + 1][3], u4_lo(w1),
                       u4_hi(w1));
            }
          }
        }
        // logits (log2 domain): c0, c1 = row lo, tokens 8t + 2tq, 8t + 2tq + 1; c2, c3 = row hi
        float lg[2][4];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const float2 sk = *reinterpret_cast<const float2*>(st + Gm::kKS + 4 * (8 * t + 2 * tq));
          const int sl = slot0 + 8 * t + 2 * tq;
          lg[t][0] = acc[t][0] * (sk.x * cq_lo);
          lg[t][1] = acc[t][1] * (sk.y * cq_lo);
          lg[t][2] = acc[t][2] * (sk.x * cq_hi);
          lg[t][3] = acc[t][3] * (sk.y * cq_hi);
          if (!full) {
            if (sl >= lim_lo) lg[t][0] = -INFINITY;
            if (sl + 1 >= lim_lo) lg[t][1] = -INFINITY;
            if (sl >= lim_hi) lg[t][2] = -INFINITY;
            if (sl + 1 >= lim_hi) lg[t][3] = -INFINITY;
          }
        }
        if (PASS == 0) {
          const float t_lo = fmaxf(fmaxf(lg[0][0], lg[0][1]), fmaxf(lg[1][0], lg[1][1]));
          const float t_hi = fmaxf(fmaxf(lg[0][2], lg[0][3]), fmaxf(lg[1][2], lg[1][3]));
          if (__any_sync(0xffffffffu, t_lo > m_lo + kCtxLazy || t_hi > m_hi + kCtxLazy)) {
            float x_lo = t_lo, x_hi = t_hi;
            x_lo = fmaxf(x_lo, __shfl_xor_sync(0xffffffffu, x_lo, 1));
            x_lo = fmaxf(x_lo, __shfl_xor_sync(0xffffffffu, x_lo, 2));
            x_hi = fmaxf(x_hi, __shfl_xor_sync(0xffffffffu, x_hi, 1));
            x_hi = fmaxf(x_hi, __shfl_xor_sync(0xffffffffu, x_hi, 2));
            const float n_lo = fmaxf(m_lo, x_lo), n_hi = fmaxf(m_hi, x_hi);
            l_lo *= fast_exp2(m_lo - n_lo);
            l_hi *= fast_exp2(m_hi - n_hi);
            m_lo = n_lo;
            m_hi = n_hi;
          }
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            l_lo += fast_exp2(lg[t][0] - m_lo) + fast_exp2(lg[t][1] - m_lo);
            l_hi += fast_exp2(lg[t][2] - m_hi) + fast_exp2(lg[t][3] - m_hi);
          }
        } else {
          // final probabilities; the PV operand p * scale_v * 2^-E
          float pr[2][4];
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            pr[t][0] = fast_exp2(lg[t][0] - M_lo) * iL_lo;
            pr[t][1] = fast_exp2(lg[t][1] - M_lo) * iL_lo;
            pr[t][2] = fast_exp2(lg[t][2] - M_hi) * iL_hi;
            pr[t][3] = fast_exp2(lg[t][3] - M_hi) * iL_hi;
            cs_t[2 * t] = pr[t][0] + pr[t][2];
            cs_t[2 * t + 1] = pr[t][1] + pr[t][3];
          }
          float2 sv[2];
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            sv[t] = *reinterpret_cast<const float2*>(st + Gm::kVS + 4 * (8 * t + 2 * tq));
            if (!full) {  // slots past the sequence carry stale scales
              const int sl = slot0 + 8 * t + 2 * tq;
              if (sl >= L.S1) sv[t].x = 0.0f;
              if (sl + 1 >= L.S1) sv[t].y = 0.0f;
            }
          }
          const float svl = fmaxf(fmaxf(sv[0].x, sv[0].y), fmaxf(sv[1].x, sv[1].y));
          if (__any_sync(0xffffffffu, svl > sv_hi || (!e_set && svl > 0.0f))) {
            float svm = svl;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) svm = fmaxf(svm, __shfl_xor_sync(0xffffffffu, svm, o));
            const int nE = min(max(exponent_of(svm), -126), 126);
            const int dE = E - nE;
            const float f = dE >= -126 ? pow2i(min(dE, 127)) : 0.0f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              oacc[j][0] *= f;
              oacc[j][1] *= f;
              oacc[j][2] *= f;
              oacc[j][3] *= f;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) osum[j] *= f;
            E = nE;
            e_set = true;
            sv_hi = pow2i(min(E + 4, 127));
            inv2E = pow2i(-E);
          }
          // A operand of PV: tokens on K (S tile 0 then tile 1), rows on M
          uint32_t pa[4];
          pa[0] = pack_half2(pr[0][0] * sv[0].x * inv2E, pr[0][1] * sv[0].y * inv2E);
          pa[1] = pack_half2(pr[0][2] * sv[0].x * inv2E, pr[0][3] * sv[0].y * inv2E);
          pa[2] = pack_half2(pr[1][0] * sv[1].x * inv2E, pr[1][1] * sv[1].y * inv2E);
          pa[3] = pack_half2(pr[1][2] * sv[1].x * inv2E, pr[1][3] * sv[1].y * inv2E);
          // O += P V: N-tile j holds head dims D(j, n) = 16 n + j (n the B
          // column, lane g supplies column g); V rows 2tq, 2tq+1 (k 2tq, 2tq+1)
          // and 2tq+8, 2tq+9 (k 2tq+8, 2tq+9)
          if (BITS == 8) {
            const uint4 va = *reinterpret_cast<const uint4*>(st + voff[0]);
            const uint4 vb = *reinterpret_cast<const uint4*>(st + voff[1]);
            const uint4 vc = *reinterpret_cast<const uint4*>(st + voff[2]);
            const uint4 vd = *reinterpret_cast<const uint4*>(st + voff[3]);
            const uint32_t xa[4] = {va.x, va.y, va.z, va.w}, xb[4] = {vb.x, vb.y, vb.z, vb.w};
            const uint32_t xc[4] = {vc.x, vc.y, vc.z, vc.w}, xd[4] = {vd.x, vd.y, vd.z, vd.w};
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int wd = j >> 2, by = j & 3;
              uint32_t b0, b1;
              if (FP8) {
                b0 = e4m3_pair_to_h2(xa[wd], xb[wd], by);
                b1 = e4m3_pair_to_h2(xc[wd], xd[wd], by);
              } else {
                const uint32_t sel = (uint32_t)by | ((uint32_t)(4 + by) << 8);
                b0 = u8_even(prmt(xa[wd], xb[wd], sel));
                b1 = u8_even(prmt(xc[wd], xd[wd], sel));
              }
              mma16816(oacc[j], pa[0], pa[1], pa[2], pa[3], b0, b1);
            }
          } else {
            const uint2 va = *reinterpret_cast<const uint2*>(st + voff[0]);
            const uint2 vb = *reinterpret_cast<const uint2*>(st + voff[1]);
            const uint2 vc = *reinterpret_cast<const uint2*>(st + voff[2]);
            const uint2 vd = *reinterpret_cast<const uint2*>(st + voff[3]);
            const uint32_t xa[2] = {va.x, va.y}, xb[2] = {vb.x, vb.y}, xc[2] = {vc.x, vc.y}, xd[2] = {vd.x, vd.y};
#pragma unroll
            for (int u = 0; u < 2; ++u) {
#pragma unroll
              for (int mm = 0; mm < 2; ++mm) {
                // bytes 2mm, 2mm+1 of word u: head dims 16g + 8u + 4mm + {0..3}
                const uint32_t sel = mm == 0 ? 0x5410u : 0x7632u;
                const uint32_t pab = prmt(xa[u], xb[u], sel), pcd = prmt(xc[u], xd[u], sel);
                const uint32_t pab2 = pab >> 8, pcd2 = pcd >> 8;
                const int j0 = 8 * u + 4 * mm;
                mma16816(oacc[j0 + 0], pa[0], pa[1], pa[2], pa[3], u4_lo(pab), u4_lo(pcd));
                mma16816(oacc[j0 + 1], pa[0], pa[1], pa[2], pa[3], u4_hi(pab), u4_hi(pcd));
                mma16816(oacc[j0 + 2], pa[0], pa[1], pa[2], pa[3], u4_lo(pab2), u4_lo(pcd2));
                mma16816(oacc[j0 + 3], pa[0], pa[1], pa[2], pa[3], u4_hi(pab2), u4_hi(pcd2));
              }
            }
          }
          if (kOffset) {
            constexpr uint32_t kOne = 0x3C003C00u;  // fp16 (1, 1)
            mma16816(osum, pa[0], pa[1], pa[2], pa[3], kOne, kOne);
          }
        }
      }
      if (PASS == 1) {
        // this warp's column sums of page p: over the lane's two rows, then
        // over the 8 row groups; lanes 0..3 hold tokens 2tq, 2tq+1, 8+2tq, 9+2tq
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          cs_t[u] += __shfl_xor_sync(0xffffffffu, cs_t[u], 4);
          cs_t[u] += __shfl_xor_sync(0xffffffffu, cs_t[u], 8);
          cs_t[u] += __shfl_xor_sync(0xffffffffu, cs_t[u], 16);
        }
        if (g == 0) {
          float* cw = sh_cs[p & 1][warp];
          cw[2 * tq] = cs_t[0];
          cw[2 * tq + 1] = cs_t[1];
          cw[8 + 2 * tq] = cs_t[2];
          cw[9 + 2 * tq] = cs_t[3];
        }
      }
    }
    cp_async_wait<0>();
    __syncthreads();
    if (PASS == 1 && npages > 0 && threadIdx.x < 16) {
      const int slot = (npages - 1) * kPage + threadIdx.x;
      if (slot < L.S1) {
        const int pb = (npages - 1) & 1;
        float v = sh_cs[pb][0][threadIdx.x];
#pragma unroll
        for (int w2 = 1; w2 < kCtxWarps; ++w2) v += sh_cs[pb][w2][threadIdx.x];
        colsum[kSinks + slot] = round == 0 ? v : colsum[kSinks + slot] + v;
      }
    }
    if (PASS == 1 && round == 0) {
      // slots no row of this CTA sees get a zero column sum (the reduction
      // reads every slot of every CTA's row)
      for (int sl = npages * kPage + threadIdx.x; sl < L.S1; sl += kCtxThreads) colsum[kSinks + sl] = 0.0f;
    }

    // ---- the bf16 window (hybrid precision): tiles of 16 positions from
    // rlo, K and V exact in bf16 (bf16 MMA; the query rows again as bf16 A
    // fragments, q' = q 2^e being exact in bf16 too)
    if (WIN && nrt > 0) {
      const int W = s.ring;
      uint32_t qb[8][4];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int row = rr ? r_hi : r_lo;
        const bool ok = (rr ? ok_hi : ok_lo) && active;
        const uint16_t* qrow =
            a.q + (((size_t)bl * s.hq + h * G + (ok ? row % G : 0)) * n + (ok ? row / G : 0)) * kHeadDim;
        const float f2e = pow2i(e_row[rr]);
#pragma unroll
        for (int st = 0; st < 8; ++st) {
          const int d0 = 16 * st + 2 * tq, d1 = d0 + 8;
          float x0 = 0.0f, x1 = 0.0f, x2 = 0.0f, x3 = 0.0f;
          if (ok) {
            const uint32_t w0 = *reinterpret_cast<const uint32_t*>(qrow + d0);
            const uint32_t w1 = *reinterpret_cast<const uint32_t*>(qrow + d1);
            x0 = bf16f(w0 & 0xFFFFu) * f2e;
            x1 = bf16f(w0 >> 16) * f2e;
            x2 = bf16f(w1 & 0xFFFFu) * f2e;
            x3 = bf16f(w1 >> 16) * f2e;
          }
          qb[st][rr] = pack_bf16x2(x0, x1);
          qb[st][2 + rr] = pack_bf16x2(x2, x3);
        }
      }
      const float cr_lo = a.qk_scale_log2 * pow2i(-e_row[0]), cr_hi = a.qk_scale_log2 * pow2i(-e_row[1]);
      const int re_lo = ok_lo ? ctx_ring_end(L, i_lo) : 0, re_hi = ok_hi ? ctx_ring_end(L, i_hi) : 0;
      // the PV operand of window tokens: p in the units of the pool's
      // accumulators (their sum is scaled by 2^24 (2^20) and 2^E at the end)
      const float rscale = pow2i(max((kOffset ? -24 : 0) - E, -126));
      const uint16_t* rk = s.ring_k + ((size_t)b * hkv + h) * W * kHeadDim;
      const uint16_t* rv = s.ring_v + ((size_t)b * hkv + h) * W * kHeadDim;
      auto ring_issue = [&](int u) {
        if (u < nrt) {
          const uint32_t sb = ring + (u & 1) * kRingStage;
          for (int c = threadIdx.x; c < (kNeedV ? 512 : 256); c += kCtxThreads) {
            const int kv = c >> 8, row = (c >> 4) & 15, ch = c & 15;
            const int pos = L.rlo + 16 * u + row;
            const uint32_t dst = sb + (uint32_t)((kv * 16 + row) * kRingRow * 2 + ch * 16);
            if (pos < L.P1)
              cp_async16_if(true, dst, (kv ? rv : rk) + (size_t)((pos - kSinks) % W) * kHeadDim + ch * 8);
            else  // past the window's end: zeros (a zero probability times stale bits could be NaN)
              asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0u) : "memory");
          }
        }
        cp_async_commit();
      };
      ring_issue(0);
#pragma unroll 1
      for (int u = 0; u < nrt; ++u) {
        ring_issue(u + 1);
        cp_async_wait<1>();
        __syncthreads();  // tile u is in; every warp is done with tile u - 1
        if (PASS == 1 && u > 0 && threadIdx.x < 16) {
          const int e2 = 16 * (u - 1) + threadIdx.x;
          if (L.rlo + e2 < L.P1) {
            const int pb = (u - 1) & 1;
            float v = sh_cs[pb][0][threadIdx.x];
#pragma unroll
            for (int w2 = 1; w2 < kCtxWarps; ++w2) v += sh_cs[pb][w2][threadIdx.x];
            cs_ring[e2] += v;
          }
        }
        const int pos0 = L.rlo + 16 * u;
        float cs_t[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (active && pos0 < wring_end) {
          const uint32_t sb = ring + (u & 1) * kRingStage;
          float acc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
          // B fragments by ldmatrix: matrices (tokens 0..7 | 8..15) x (dims 16st.. | 16st+8..)
          const int mtx = lane >> 3;
          const uint32_t kaddr = sb + (uint32_t)((((mtx >> 1) * 8 + (lane & 7)) * kRingRow + ((mtx & 1) * 8)) * 2);
#pragma unroll
          for (int st = 0; st < 8; ++st) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(b0, b1, b2, b3, kaddr + 32 * st);
            mma16816_bf16(acc[0], qb[st][0], qb[st][1], qb[st][2], qb[st][3], b0, b1);
            mma16816_bf16(acc[1], qb[st][0], qb[st][1], qb[st][2], qb[st][3], b2, b3);
          }
          float lg[2][4];
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int ps = pos0 + 8 * t + 2 * tq;
            lg[t][0] = ps < re_lo ? acc[t][0] * cr_lo : -INFINITY;
            lg[t][1] = ps + 1 < re_lo ? acc[t][1] * cr_lo : -INFINITY;
            lg[t][2] = ps < re_hi ? acc[t][2] * cr_hi : -INFINITY;
            lg[t][3] = ps + 1 < re_hi ? acc[t][3] * cr_hi : -INFINITY;
          }
          if (PASS == 0) {
            const float t_lo = fmaxf(fmaxf(lg[0][0], lg[0][1]), fmaxf(lg[1][0], lg[1][1]));
            const float t_hi = fmaxf(fmaxf(lg[0][2], lg[0][3]), fmaxf(lg[1][2], lg[1][3]));
            if (__any_sync(0xffffffffu, t_lo > m_lo + kCtxLazy || t_hi > m_hi + kCtxLazy)) {
              float x_lo = t_lo, x_hi = t_hi;
              x_lo = fmaxf(x_lo, __shfl_xor_sync(0xffffffffu, x_lo, 1));
              x_lo = fmaxf(x_lo, __shfl_xor_sync(0xffffffffu, x_lo, 2));
              x_hi = fmaxf(x_hi, __shfl_xor_sync(0xffffffffu, x_hi, 1));
              x_hi = fmaxf(x_hi, __shfl_xor_sync(0xffffffffu, x_hi, 2));
              const float n_lo = fmaxf(m_lo, x_lo), n_hi = fmaxf(m_hi, x_hi);
              l_lo *= fast_exp2(m_lo - n_lo);
              l_hi *= fast_exp2(m_hi - n_hi);
              m_lo = n_lo;
              m_hi = n_hi;
            }
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              l_lo += fast_exp2(lg[t][0] - m_lo) + fast_exp2(lg[t][1] - m_lo);
              l_hi += fast_exp2(lg[t][2] - m_hi) + fast_exp2(lg[t][3] - m_hi);
            }
          } else {
            float pr[2][4];
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              pr[t][0] = fast_exp2(lg[t][0] - M_lo) * iL_lo;
              pr[t][1] = fast_exp2(lg[t][1] - M_lo) * iL_lo;
              pr[t][2] = fast_exp2(lg[t][2] - M_hi) * iL_hi;
              pr[t][3] = fast_exp2(lg[t][3] - M_hi) * iL_hi;
              cs_t[2 * t] = pr[t][0] + pr[t][2];
              cs_t[2 * t + 1] = pr[t][1] + pr[t][3];
            }
            uint32_t ph[4], pl[4];
            split_bf16x2(pr[0][0] * rscale, pr[0][1] * rscale, ph[0], pl[0]);
            split_bf16x2(pr[0][2] * rscale, pr[0][3] * rscale, ph[1], pl[1]);
            split_bf16x2(pr[1][0] * rscale, pr[1][1] * rscale, ph[2], pl[2]);
            split_bf16x2(pr[1][2] * rscale, pr[1][3] * rscale, ph[3], pl[3]);
            // V rows 2tq, 2tq+1, 2tq+8, 2tq+9 at head dims 16g .. 16g+15
            uint32_t xr[4][8];
            const int vr[4] = {2 * tq, 2 * tq + 1, 2 * tq + 8, 2 * tq + 9};
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const uint8_t* vp = smem + (u & 1) * kRingStage + ((16 + vr[q4]) * kRingRow + 16 * g) * 2;
              const uint4 y0 = *reinterpret_cast<const uint4*>(vp);
              const uint4 y1 = *reinterpret_cast<const uint4*>(vp + 16);
              xr[q4][0] = y0.x; xr[q4][1] = y0.y; xr[q4][2] = y0.z; xr[q4][3] = y0.w;
              xr[q4][4] = y1.x; xr[q4][5] = y1.y; xr[q4][6] = y1.z; xr[q4][7] = y1.w;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
              uint32_t b0 = prmt(xr[0][j >> 1], xr[1][j >> 1], sel);
              uint32_t b1 = prmt(xr[2][j >> 1], xr[3][j >> 1], sel);
              if (kOffset && BITS == 4 && (j & 1)) {  // these N-tiles hold 16x values (INT4 high nibbles)
                b0 = bf16x2_times16(b0);
                b1 = bf16x2_times16(b1);
              }
              mma16816_bf16(oacc[j], ph[0], ph[1], ph[2], ph[3], b0, b1);
              mma16816_bf16(oacc[j], pl[0], pl[1], pl[2], pl[3], b0, b1);
            }
          }
        }
        if (PASS == 1) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            cs_t[q4] += __shfl_xor_sync(0xffffffffu, cs_t[q4], 4);
            cs_t[q4] += __shfl_xor_sync(0xffffffffu, cs_t[q4], 8);
            cs_t[q4] += __shfl_xor_sync(0xffffffffu, cs_t[q4], 16);
          }
          if (g == 0) {
            float* cw = sh_cs[u & 1][warp];
            cw[2 * tq] = cs_t[0];
            cw[2 * tq + 1] = cs_t[1];
            cw[8 + 2 * tq] = cs_t[2];
            cw[9 + 2 * tq] = cs_t[3];
          }
        }
      }
      cp_async_wait<0>();
      __syncthreads();
      if (PASS == 1 && threadIdx.x < 16) {
        const int e2 = 16 * (nrt - 1) + threadIdx.x;
        if (L.rlo + e2 < L.P1) {
          const int pb = (nrt - 1) & 1;
          float v = sh_cs[pb][0][threadIdx.x];
#pragma unroll
          for (int w2 = 1; w2 < kCtxWarps; ++w2) v += sh_cs[pb][w2][threadIdx.x];
          cs_ring[e2] += v;
        }
      }
    }

    if (PASS == 0) {
      if (active) {
        l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
        l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
        if (tq == 0) {
          const size_t srow = (size_t)pair * R;
          if (ok_lo) *reinterpret_cast<float2*>(a.stats + (srow + r_lo) * 2) = make_float2(m_lo, l_lo);
          if (ok_hi) *reinterpret_cast<float2*>(a.stats + (srow + r_hi) * 2) = make_float2(m_hi, l_hi);
        }
      }
    } else {
      // sinks: probabilities, their column sums, their V rows into the output
      float ps[2][kSinks];
#pragma unroll
      for (int sk = 0; sk < kSinks; ++sk) {
        ps[0][sk] = sk < ns_lo ? fast_exp2(sk_lg[0][sk] - M_lo) * iL_lo : 0.0f;
        ps[1][sk] = sk < ns_hi ? fast_exp2(sk_lg[1][sk] - M_hi) * iL_hi : 0.0f;
      }
      // the sink column sums of this CTA's rows: every lane of a row group has
      // the same values; lanes tq == 0 of each row group add theirs
      if (active) {
#pragma unroll
        for (int sk = 0; sk < kSinks; ++sk) {
          float v = tq == 0 ? ps[0][sk] + ps[1][sk] : 0.0f;
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) sh_sk[warp][sk] = v;
        }
      } else if (lane == 0) {
#pragma unroll
        for (int sk = 0; sk < kSinks; ++sk) sh_sk[warp][sk] = 0.0f;
      }
      __syncthreads();
      if (threadIdx.x < kSinks) {
        float v = sh_sk[0][threadIdx.x];
#pragma unroll
        for (int w2 = 1; w2 < kCtxWarps; ++w2) v += sh_sk[w2][threadIdx.x];
        colsum[threadIdx.x] = round == 0 ? v : colsum[threadIdx.x] + v;
      }
      __syncthreads();
      if (active) {
        // output rows r_lo / r_hi, head dims 32tq + j (j < 16: N-tile j, column
        // 2tq) and 32tq + 16 + j (column 2tq + 1): 64 contiguous bytes each
        const float f2E = pow2i(E);
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const int row = rr ? r_hi : r_lo;
          if (!(rr ? ok_hi : ok_lo)) continue;
          const int i = row / G, gq = row % G;
          uint16_t* orow = a.out + (((size_t)bl * s.hq + h * G + gq) * n + i) * kHeadDim + 32 * tq;
          const float bias = kOffset ? kOffV * osum[2 * rr] : 0.0f;
          uint32_t packed[16];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
              float o2[2];
#pragma unroll
              for (int jj = 0; jj < 2; ++jj) {
                const int jt = j + jj;
                // INT4: odd N-tiles carry the 16x high nibbles
                const float sc = kOffset ? (BITS == 4 && (jt & 1) ? 0x1p20f : 0x1p24f) : 1.0f;
                float o = (oacc[jt][2 * rr + half] * sc - bias) * f2E;
                const int d = 32 * tq + 16 * half + jt;
#pragma unroll
                for (int sk = 0; sk < kSinks; ++sk)
                  o = fmaf(ps[rr][sk], bf16f(sink_v[sk * kHeadDim + d]), o);
                o2[jj] = o;
              }
              const __nv_bfloat162 hv = __floats2bfloat162_rn(o2[0], o2[1]);
              packed[8 * half + j / 2] = *reinterpret_cast<const uint32_t*>(&hv);
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u)
            reinterpret_cast<uint4*>(orow)[u] =
                make_uint4(packed[4 * u], packed[4 * u + 1], packed[4 * u + 2], packed[4 * u + 3]);
        }
      }
    }
    __syncthreads();  // the ring and sh_cs are reused by the next round
  }

  if (PASS == 1 && a.accumulate) {
    // the last CTA of this (sequence, KV head) adds every CTA's column sums,
    // in CTA order, to the scores
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) sh_last = atomicAdd(&a.ticket[pair], 1) == a.groups - 1;
    __syncthreads();
    if (sh_last) {
      __threadfence();
      const float* base = a.colsum + (size_t)pair * a.groups * a.cs_row;
      if (WIN && s.ring > 0) {
        for (int e = threadIdx.x; e < L.P1 - L.rlo; e += kCtxThreads) {
          float v = 0.0f;
          for (int c = 0; c < a.groups; ++c) v += base[(size_t)c * a.cs_row + kSinks + a.s_cap + e];
          s.ring_score[((size_t)b * hkv + h) * s.ring + (L.rlo + e - kSinks) % s.ring] += v;
        }
      }
      for (int sl = threadIdx.x; sl < kSinks + L.S1; sl += kCtxThreads) {
        if (sl < kSinks && sl >= n_sinks) continue;
        float v = 0.0f;
        for (int c = 0; c < a.groups; ++c) v += base[(size_t)c * a.cs_row + sl];
        if (sl < kSinks) {
          s.sink_score[((size_t)b * hkv + h) * kSinks + sl] += v;
        } else {
          const int slot = sl - kSinks;
          const int blk = blk_of(slot / kPage);
          if ((unsigned)blk < (unsigned)s.num_blocks) s.score[((size_t)blk * hkv + h) * kPage + slot % kPage] += v;
        }
      }
    }
  }
}

template <int BITS, bool FP8, int PASS, bool WIN>
cudaError_t launch_ctx_t(const DevState& s, int seq_begin, int batch, const CtxArgs& a, cudaStream_t st) {
  using Gm = CtxGeom<BITS>;
  const int ring_bytes = WIN && 2 * kRingStage > kCtxStages * Gm::kStage ? 2 * kRingStage : kCtxStages * Gm::kStage;
  const int smem = ring_bytes + kCtxBtStage * 4;
  static int done[64] = {0};
  const cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(ctx_attn_kernel<BITS, FP8, PASS, WIN>), smem, done);
  if (e != cudaSuccess) return e;
  dim3 grid(a.groups, batch * s.hkv);
  ctx_attn_kernel<BITS, FP8, PASS, WIN><<<grid, kCtxThreads, smem, st>>>(s, seq_begin, a);
  return cudaGetLastError();
}

template <int BITS, bool FP8, bool WIN>
cudaError_t launch_ctx_passes(const DevState& s, int seq_begin, int batch, const CtxArgs& a, cudaStream_t st) {
  cudaError_t e = launch_ctx_t<BITS, FP8, 0, WIN>(s, seq_begin, batch, a, st);
  if (e == cudaSuccess) e = launch_ctx_t<BITS, FP8, 1, WIN>(s, seq_begin, batch, a, st);
  return e;
}

template <int BITS, bool FP8>
cudaError_t launch_ctx_codes(const DevState& s, int seq_begin, int batch, const CtxArgs& a, cudaStream_t st) {
  return s.ring > 0 ? launch_ctx_passes<BITS, FP8, true>(s, seq_begin, batch, a, st)
                    : launch_ctx_passes<BITS, FP8, false>(s, seq_begin, batch, a, st);
}

}  // namespace

int ctx_groups(int n, int group) {
  const int mtiles = (n * group + 15) / 16;
  const int g = (mtiles + kCtxWarps - 1) / kCtxWarps;
  return g < kMaxCtxGroups ? g : kMaxCtxGroups;
}

cudaError_t launch_ctx_attention(const DevState& s, int seq_begin, int batch, int n, const uint16_t* q,
                                 uint16_t* out, float* stats, float* colsum, int* ticket, int s_cap,
                                 float qk_scale_log2, bool accumulate, cudaStream_t st) {
  CtxArgs a;
  a.q = q;
  a.out = out;
  a.stats = stats;
  a.colsum = colsum;
  a.ticket = ticket;
  a.n = n;
  a.groups = ctx_groups(n, s.group);
  a.s_cap = s_cap;
  a.cs_row = kSinks + s_cap + s.ring;
  a.qk_scale_log2 = qk_scale_log2;
  a.accumulate = accumulate ? 1 : 0;
  cudaError_t e;
  if (s.bits == 8 && s.fp8)
    e = launch_ctx_codes<8, true>(s, seq_begin, batch, a, st);
  else if (s.bits == 8)
    e = launch_ctx_codes<8, false>(s, seq_begin, batch, a, st);
  else
    e = launch_ctx_codes<4, false>(s, seq_begin, batch, a, st);
  return e;
}

}  // namespace kvc
