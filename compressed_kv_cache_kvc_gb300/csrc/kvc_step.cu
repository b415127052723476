// The decode-step work that follows the split-K attention, in two kernels.
//
// step_post_kernel, one CTA per (KV head, sequence): merge of the partials
// with the sinks (bf16 outputs), H2O score accumulation, kept-set selection
// and the compaction move lists.  It computes exactly what attn_merge_kernel
// + select_kernel + the list phase of compact_kernel compute, in the same
// order, but the scores, keys, positions and keep decisions stay in shared
// memory between the phases.  The page prefix of the slice comes from the
// split kernel, so no CTA reads another sequence's length; the last of a
// sequence's KV-head CTAs to finish (an atomic ticket: no CTA waits for
// another) applies its new length and releases its pages.  Released pages
// are only taken by later calls, after step_moves_kernel has read them.
//
// With block-granular eviction the post kernel stops after the scores; the
// page keys and the eviction follow as launches of their own (kvc_select.cu).
//
// step_moves_kernel, one CTA per (KV head, sequence): the row moves of the
// lists.  Moves run in a launch of their own because, sharing an SM with
// another CTA's selection phase, their global-memory traffic stalls that
// phase's shared-memory work; when no pair moves more than kInlineMoves rows
// (the steady state moves one), the post kernel moves them and the move
// kernel is not launched.
//
// (Technical Report: KV Cache Compression for Text-Only LLMs, sections 3.3
// and 3.4; "KV Cache optimization techniques" sections 2.2, 2.4 and 3.2.)
#include <algorithm>
#include <type_traits>

#include "kvc_device.h"
#include "kvc_internal.h"
#include "kvc_mma.h"  // codes::smem_u32

namespace kvc {
namespace {

using namespace dev;

constexpr int kStepThreads = 512;
constexpr int kStepBtStage = 2048;

// Predicated stores and shared-memory adds (no branch).
__device__ __forceinline__ void st4_if(bool pred, float* dst, float a, float b, float c, float d) {
  asm volatile(
      "{\n .reg .pred q;\n setp.ne.u32 q, %0, 0;\n"
      " @q st.global.v4.f32 [%1], {%2, %3, %4, %5};\n}\n" ::"r"((uint32_t)pred),
      "l"(dst), "f"(a), "f"(b), "f"(c), "f"(d)
      : "memory");
}
__device__ __forceinline__ void st1_if(bool pred, float* dst, float a) {
  asm volatile(
      "{\n .reg .pred q;\n setp.ne.u32 q, %0, 0;\n"
      " @q st.global.f32 [%1], %2;\n}\n" ::"r"((uint32_t)pred),
      "l"(dst), "f"(a)
      : "memory");
}
__device__ __forceinline__ void red_shared_add_if(bool pred, int* addr, int v) {
  asm volatile(
      "{\n .reg .pred q;\n setp.ne.u32 q, %0, 0;\n"
      " @q red.shared.add.s32 [%1], %2;\n}\n" ::"r"((uint32_t)pred),
      "r"(codes::smem_u32(addr)), "r"(v)
      : "memory");
}

// NT threads: 512 (two CTAs per SM) or, when the pairs are no more than the
// SMs, 1024 (one pair per SM, twice the threads on its slots).
template <int NT, int GC>
__global__ void __launch_bounds__(NT, 1024 / NT) step_post_kernel(DevState s, int seq_begin, int batch,
                                                                const uint16_t* __restrict__ q,
                                                                uint16_t* __restrict__ out, float qk_scale_log2,
                                                                AttnWork w, StepArgs a) {
  __shared__ MergeShared ms;
  __shared__ int32_t sh_bt[kStepBtStage];
  __shared__ int hist[kRadixBins];
  __shared__ int sh_sel[3];
  __shared__ int sh_warp[32];
  extern __shared__ __align__(16) uint32_t dyn[];

  const int h = blockIdx.x;
  const int bl = blockIdx.y;
  const int b = seq_begin + bl;
  // mode 0: H2O; 1: StreamingLLM (no scores); 2: block-granular eviction
  // (scores only: the page selection runs in launches of its own)
  const bool block = a.mode == 2;
  const bool h2o = a.mode != 1;
  const int hkv = s.hkv;
  const int G = s.group;
  const int S = s.seq_slots[b];
  const size_t pair = (size_t)bl * hkv + h;
  // the selection's first radix histogram is built by the score pass
  for (int i = threadIdx.x; i < kRadixBins; i += blockDim.x) hist[i] = 0;
  const int32_t* bt = s.block_table + (size_t)b * s.max_bps;
  const int npages = (S + kPage - 1) / kPage;
  const int32_t* btp = bt;
  if (npages <= kStepBtStage) {
    for (int i = threadIdx.x; i < npages; i += blockDim.x) sh_bt[i] = bt[i];
    btp = sh_bt;
  }
  // the host sized the shared key buffer from its mirror of the lengths; a
  // longer sequence on the device (state restored without a host resync) is
  // flagged and keeps its slots
  const bool fits = a.smem_slots == 0 || S <= a.smem_slots;
  uint32_t* keys;
  int32_t* pos;
  if (a.smem_slots > 0) {
    keys = dyn;
    pos = a.pos_smem ? reinterpret_cast<int32_t*>(dyn + a.smem_slots) : a.g_pos + pair * a.s_cap;
  } else {
    keys = a.g_keys + pair * a.s_cap;
    pos = a.g_pos + pair * a.s_cap;
  }
  if (a.merged) {
    // the merge ran on the attention's stream (kvc_decode_step_overlap):
    // its per-head (M, L), and 1 / L as the merge forms it
    if ((int)threadIdx.x < G) {
      const float* st = w.stats + ((size_t)bl * s.hq + h * G + threadIdx.x) * 2;
      const float L = st[1];
      ms.M[threadIdx.x] = st[0];
      ms.invL[threadIdx.x] = L > 0.0f ? 1.0f / L : 0.0f;
    }
    __syncthreads();  // publishes ms and the block-table row
  } else {
    // (the merge's barriers publish the block-table row)
    merge_phase(s, seq_begin, batch, w.cum, h, bl, q, out, qk_scale_log2, w, h2o, ms);
  }
  if (h2o) ring_score_pass(s, w, seq_begin + bl, bl, h, ms);

  const int P = s.seq_pos[b];
  const int ns = min(P, kSinks);
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
  if (h == 0 && threadIdx.x == 0 && !block) {
    s.plan[2 * b] = S;
    s.plan[2 * b + 1] = n_keep;
  }

  __syncthreads();

  // ---- scores (H2O) and selection keys.  Keys: 0xFFFFFFFF for the recent
  // window (always kept), else the fp32 score bits (H2O) or 0 (StreamingLLM).
  // Four consecutive slots (a quarter page) per thread and round, moved as
  // 16-byte vectors; every load of a round (the group's logit vectors, the
  // positions and scores) is issued before the first use.  The pass is bound
  // by instruction issue, so the round is branch-free: a bad block id loads
  // from block 0 and is masked, the stores and histogram adds are
  // predicated, and the ragged last quarter page runs after the loop.
  constexpr int GL = GC > 0 ? GC : kMaxGroup;  // logit rows held per round
  const int Gr = GC > 0 ? GC : G;
  const float* lgr = w.logits + pair * G * w.s_cap;
  // whole 128-byte lines of logits (rows 128-byte aligned) can be dropped
  const bool discard_ok = h2o && (w.s_cap % 32) == 0 && ((uintptr_t)lgr % 128) == 0;
  const bool want_keys = !block && fits;
  // the group's (M, 1/L) in registers when they fit beside the logit rows
  constexpr bool kStatsInRegs = GL <= 5;
  float Mg[GL], iLg[GL];
#pragma unroll
  for (int g = 0; g < GL; ++g) {
    Mg[g] = g < Gr ? ms.M[g] : 0.0f;
    iLg[g] = g < Gr ? ms.invL[g] : 0.0f;
  }
  int n_top = 0;   // recent-window keys of this thread (the histogram's top bin)
  bool bad = false;
  auto quad = [&](int j, auto tail_tag) {
    constexpr bool kTail = decltype(tail_tag)::value;
    const int t = 4 * j;
    const int blk = btp[t / kPage];
    const bool ok = (unsigned)blk < (unsigned)s.num_blocks;
    bad |= !ok;
    const size_t idx = ((size_t)(ok ? blk : 0) * hkv + h) * kPage + (t % kPage);
    // logit rows in chunks of at most 5 (wider groups would spill)
    constexpr int CH = GL <= 5 ? GL : 4;
    float4 lg[CH];
    auto load_rows = [&](int g0) {
#pragma unroll
      for (int i = 0; i < CH; ++i)
        lg[i] = g0 + i < Gr ? *reinterpret_cast<const float4*>(lgr + (size_t)(g0 + i) * w.s_cap + t)
                            : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    };
    if (h2o) load_rows(0);
    int4 p4 = *reinterpret_cast<const int4*>(s.slot_pos + idx);
    float4 sc4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (h2o) sc4 = *reinterpret_cast<const float4*>(s.score + idx);
    if (!ok) {
      p4 = make_int4(-1, -1, -1, -1);
      sc4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    const int pp[4] = {p4.x, p4.y, p4.z, p4.w};
    float vv[4] = {sc4.x, sc4.y, sc4.z, sc4.w};
    uint32_t kk[4];
    if (h2o) {
      // the H2O increment: sum over the group of the slot's probability, in
      // query-head order (as h2o_increment)
      float inc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int g0 = 0; g0 < GL; g0 += CH) {
        if (g0 > 0) load_rows(g0);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int i = 0; i < CH; ++i) {
            const int g = g0 + i;
            const float l = c == 0 ? lg[i].x : c == 1 ? lg[i].y : c == 2 ? lg[i].z : lg[i].w;
            const float Mv = kStatsInRegs ? Mg[g] : ms.M[g];
            const float iLv = kStatsInRegs ? iLg[g] : ms.invL[g];
            if (g < Gr) inc[c] = __fmaf_rn(fast_exp2(l - Mv), iLv, inc[c]);
          }
        }
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) vv[c] += inc[c];
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t key = h2o ? __float_as_uint(fmaxf(vv[c], 0.0f)) : 0u;
      kk[c] = ok ? (pp[c] >= thr ? 0xFFFFFFFFu : key) : 0u;
    }
    if (h2o) {
      if (kTail) {
#pragma unroll
        for (int c = 0; c < 4; ++c) st1_if(ok && t + c < S, s.score + idx + c, vv[c]);
      } else {
        st4_if(ok, s.score + idx, vv[0], vv[1], vv[2], vv[3]);
      }
    }
    if (discard_ok && !kTail) {
      // the logits of 32 slots are read once the 8 threads of their line have
      // used them: drop those lines from L2 without writing them back
      __syncwarp(__activemask());
      if ((threadIdx.x & 7) == 0 && t + 32 <= S)
#pragma unroll
        for (int g = 0; g < GL; ++g)
          if (g < Gr) asm volatile("discard.global.L2 [%0], 128;" ::"l"(lgr + (size_t)g * w.s_cap + t) : "memory");
    }
    if (!want_keys) return;
    // slots past S in the last quarter page get keys too: nothing reads them
    *reinterpret_cast<uint4*>(keys + t) = make_uint4(kk[0], kk[1], kk[2], kk[3]);
    *reinterpret_cast<int4*>(pos + t) = p4;
    // first-pass histogram (bits 31..21) of the selection; the recent
    // window's keys all fall in the top bin and are counted apart
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const bool in = !kTail || t + c < S;
      const bool top = kk[c] == 0xFFFFFFFFu;
      n_top += (in && top) ? 1 : 0;
      red_shared_add_if(in && !top, &hist[kk[c] >> 21], 1);
    }
  };
  const int nq_full = S >> 2;
  for (int j = threadIdx.x; j < nq_full; j += NT) quad(j, std::false_type());
  if ((S & 3) != 0 && (int)threadIdx.x == nq_full % NT) quad(nq_full, std::true_type());
  if (want_keys) {
    n_top = __reduce_add_sync(0xffffffffu, n_top);
    if ((threadIdx.x & 31) == 0 && n_top > 0) atomicAdd(&hist[kRadixBins - 1], n_top);
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(&s.counters[kCtrStatus], kDevBadBlockId);
  if (block) return;
  if (!fits) {  // every CTA of the sequence takes this exit (same S)
    if (threadIdx.x == 0) {
      a.n_moves[pair] = 0;
      atomicOr(&s.counters[kCtrStatus], kDevStaleHost);
    }
    return;
  }
  __syncthreads();
  bool lists_ok = true;
  if (!keep_all) {

  // ---- selection: the n_keep largest keys, ties at the threshold to the
  // lower positions
  uint32_t theta = 0xFFFFFFFFu, pos_cut = 0xFFFFFFFFu;
  if (n_keep > 0 && S - n_keep == 1) {
    // one slot goes (the steady state): the least key, and among equal least
    // keys the highest position, is the one the rule below evicts.  One
    // block-wide minimum of (key, ~position); pool positions are >= 4.
    __shared__ unsigned long long sh_min[32];
    unsigned long long best = ~0ull;
    for (int t = threadIdx.x; t < S; t += NT) {
      const unsigned long long v = ((unsigned long long)keys[t] << 32) | (uint32_t)~(uint32_t)pos[t];
      best = v < best ? v : best;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
      best = y < best ? y : best;
    }
    if ((threadIdx.x & 31) == 0) sh_min[threadIdx.x >> 5] = best;
    __syncthreads();
    best = ~0ull;
#pragma unroll
    for (int j = 0; j < NT / 32; ++j) best = sh_min[j] < best ? sh_min[j] : best;
    theta = (uint32_t)(best >> 32);
    pos_cut = ~(uint32_t)best - 1u;  // every other slot with key theta sits lower
  } else if (n_keep > 0) {
    int need, ties;
    theta = radix_select<NT>(
        S, n_keep, true, [&](int) { return true; }, [&](int i) { return keys[i]; }, hist, sh_warp, sh_sel, &need,
        &ties, /*pass0_ready=*/true);
    if (ties > need) {  // ties at theta: the lowest positions win
      int rem2, t2;
      pos_cut = radix_select<NT>(
          S, need, false, [&](int i) { return keys[i] == theta; }, [&](int i) { return (uint32_t)pos[i]; },
          hist, sh_warp, sh_sel, &rem2, &t2);
    }
  }
  const int np = n_keep;

  // ---- compaction lists.  A tile is 16 x 32 consecutive slots per warp;
  // lane l of warp w decides slots tile0 + 512 w + 32 i + l.  Holes and
  // sources are ranked in slot order (warp totals, then ballots) and go to
  // the pair's rows of the workspace key/position arrays.  Where the keys
  // and positions themselves live there, the lists overwrite them in place:
  // the i-th hole (or source) lies at a slot >= i, and every read of a tile
  // precedes its writes.
  int32_t* holes = reinterpret_cast<int32_t*>(a.g_keys + pair * a.s_cap);
  int32_t* srcs = a.g_pos + pair * a.s_cap;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t lt = (1u << lane) - 1u;
  const int wlo = keep_window(S, np);
  int hole_base = 0, src_base = 0;
  for (int tile0 = 0; tile0 < S; tile0 += NT * 16) {
    const int wbase = tile0 + warp * 512 + lane;
    uint32_t hole_bits = 0, src_bits = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int t = wbase + 32 * i;
      if (t < S) {
        const uint32_t k = keys[t];
        const bool kept = n_keep > 0 && (k > theta || (k == theta && (uint32_t)pos[t] <= pos_cut));
        const bool inwin = (unsigned)(t - wlo) < (unsigned)max(np, 0);
        if (kept && !inwin) src_bits |= 1u << i;
        if (!kept && inwin) hole_bits |= 1u << i;
      }
    }
    const uint32_t packed = __reduce_add_sync(0xffffffffu, __popc(hole_bits) | (__popc(src_bits) << 16));
    if (lane == 0) sh_warp[warp] = (int)packed;
    __syncthreads();
    int before = 0, tot = 0;
#pragma unroll
    for (int j = 0; j < NT / 32; ++j) {
      const int v = sh_warp[j];
      before += j < warp ? v : 0;
      tot += v;
    }
    int ph = hole_base + (before & 0xFFFF), ps = src_base + (before >> 16);
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
      const uint32_t mh = __ballot_sync(0xffffffffu, (hole_bits >> i) & 1u);
      const uint32_t msk = __ballot_sync(0xffffffffu, (src_bits >> i) & 1u);
      if ((mh | msk) == 0u) continue;
      const int t = wbase + 32 * i;
      if ((hole_bits >> i) & 1u) holes[ph + __popc(mh & lt)] = slot_index(s, btp, t, h);
      if ((src_bits >> i) & 1u) srcs[ps + __popc(msk & lt)] = slot_index(s, btp, t, h);
      ph += __popc(mh);
      ps += __popc(msk);
    }
    hole_base += tot & 0xFFFF;
    src_base += tot >> 16;
    __syncthreads();
  }
  if (hole_base != src_base) {
    if (threadIdx.x == 0) atomicOr(&s.counters[kCtrStatus], kDevBadKeepMask);
    lists_ok = false;
  }

  if (threadIdx.x == 0) a.n_moves[pair] = lists_ok ? hole_base : 0;
  if (a.inline_moves && lists_ok && hole_base > 0) {
    // few rows (no move kernel follows): this CTA moves them (the lists are
    // this CTA's own writes, visible after the barrier)
    __syncthreads();
    move_rows(s, holes, srcs, hole_base);
  }

  } else if (threadIdx.x == 0) {
    a.n_moves[pair] = 0;
  }

  // ---- the last of the sequence's KV-head CTAs to finish applies its new
  // length and releases its pages past ceil(n'/16) (every CTA of the
  // sequence has the same S and n_keep)
  __shared__ int sh_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    sh_last = atomicAdd(&w.seq_ticket[bl], 1) == hkv - 1;
  }
  __syncthreads();
  if (!sh_last) return;
  __threadfence();
  const int keep_pages = (n_keep + kPage - 1) / kPage;
  const int nfree = npages - keep_pages;
  const int p0 = keep_window(S, n_keep) / kPage;  // first page of the window
  if (threadIdx.x == 0) {
    int fbase = -1;
    if (nfree > 0) {
      fbase = atomicAdd(&s.counters[kCtrFreeTop], nfree);
      if (fbase + nfree > s.num_blocks) {
        atomicSub(&s.counters[kCtrFreeTop], nfree);
        atomicOr(&s.counters[kCtrStatus], kDevStackOverflow);
        fbase = -1;
      }
    }
    sh_sel[0] = fbase;
    if (n_keep < S) s.seq_slots[b] = n_keep;
    w.seq_ticket[bl] = 0;
  }
  __syncthreads();
  const int fbase = sh_sel[0];
  // released: pages [0, p0) and [p0 + keep_pages, npages) of the old row
  if (fbase >= 0)
    for (int j = threadIdx.x; j < nfree; j += blockDim.x) s.free_stack[fbase + j] = btp[j < p0 ? j : keep_pages + j];
  if (p0 > 0) shift_row(s.block_table + (size_t)b * s.max_bps, p0, keep_pages);
}

// Row moves of one (KV head, sequence) per CTA (see move_rows).
// With fewer pairs than SMs, gridDim.z CTAs share a pair's lists, each a
// contiguous share.
__global__ void __launch_bounds__(kStepThreads, 2) step_moves_kernel(DevState s, StepArgs a) {
  const size_t pair = (size_t)blockIdx.y * s.hkv + blockIdx.x;
  const int n = a.n_moves[pair];
  const int lo = (int)((long long)n * blockIdx.z / gridDim.z);
  const int hi = (int)((long long)n * (blockIdx.z + 1) / gridDim.z);
  move_rows(s, reinterpret_cast<const int32_t*>(a.g_keys + pair * a.s_cap) + lo, a.g_pos + pair * a.s_cap + lo,
            hi - lo);
}

}  // namespace

int step_max_smem_bytes() { return 160 * 1024; }

template <int NT, int GC>
cudaError_t launch_step_post_nt(const DevState& s, int seq_begin, int batch, const uint16_t* q, uint16_t* out,
                                float qk_scale_log2, const AttnWork& w, const StepArgs& a, cudaStream_t st) {
  const int smem = a.smem_slots > 0 ? a.smem_slots * (a.pos_smem ? 8 : 4) : 0;
  if (smem > 0) {
    static int done[64] = {0};
    const cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(step_post_kernel<NT, GC>), step_max_smem_bytes(), done);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(s.hkv, batch);
  step_post_kernel<NT, GC><<<grid, NT, smem, st>>>(s, seq_begin, batch, q, out, qk_scale_log2, w, a);
  return cudaGetLastError();
}

cudaError_t launch_step_post(const DevState& s, int seq_begin, int batch, const uint16_t* q, uint16_t* out,
                             float qk_scale_log2, const AttnWork& w, const StepArgs& a, int sm_count,
                             cudaStream_t st) {
  // the group sizes of common layouts get a score pass of their own width
  // (1: multi-head attention; 4 and 5: GQA); others take the general one
  const bool wide = batch * s.hkv <= sm_count;
  switch (s.group) {
#define KVC_POST_CASE(GC)                                                                              \
  case GC:                                                                                             \
    return wide ? launch_step_post_nt<1024, GC>(s, seq_begin, batch, q, out, qk_scale_log2, w, a, st) \
                : launch_step_post_nt<kStepThreads, GC>(s, seq_begin, batch, q, out, qk_scale_log2, w, a, st);
    KVC_POST_CASE(1)
    KVC_POST_CASE(4)
    KVC_POST_CASE(5)
#undef KVC_POST_CASE
    default:
      return wide ? launch_step_post_nt<1024, 0>(s, seq_begin, batch, q, out, qk_scale_log2, w, a, st)
                  : launch_step_post_nt<kStepThreads, 0>(s, seq_begin, batch, q, out, qk_scale_log2, w, a, st);
  }
}

cudaError_t launch_step_moves(const DevState& s, int batch, const StepArgs& a, int sm_count, int max_moves,
                              cudaStream_t st) {
  // with fewer pairs than SMs, up to two CTAs per SM in all, but no CTA with
  // fewer than ~256 moves (at steady state a pair moves one row)
  const int pairs = batch * s.hkv;
  int z = pairs < sm_count ? (2 * sm_count + pairs - 1) / pairs : 1;
  z = std::max(1, std::min(z, (max_moves + 255) / 256));
  dim3 grid(s.hkv, batch, z);
  step_moves_kernel<<<grid, kStepThreads, 0, st>>>(s, a);
  return cudaGetLastError();
}

}  // namespace kvc
