// Split-K paged decode attention with the dequantisation fused into QK^T and
// PV, and the online-softmax merge with the bf16 attention sinks and the H2O
// score accumulation.
//
// The method: out = softmax(q K^T / sqrt(d)) V (Technical Report, section
// 1.1), where the pool's keys and values are code * scale (section 3.2, "scores
// = Q @ (K_q * scale_k).T / sqrt(d); out = softmax(scores) @ (V_q * scale_v)")
// and the four sinks are bf16 (section 3.2).  H2O adds each token's softmax
// probability, summed over the query heads of its KV head, to its score
// (section 3.4).
//
// GB300 design
//   * Stream-K grid: one wave of resident CTAs; the pages of all (sequence,
//     KV head) pairs are laid end to end and every CTA takes an equal run
//     (which may span a pair boundary: one partial per pair touched).  Inside
//     a CTA the 4 warps take the run's pages round-robin.
//   * Each warp streams its pages through a private ring of shared-memory
//     stages with cp.async: a K or V page of one head is one contiguous
//     2 KB (8-bit) / 1 KB (INT4) run of the pool, copied by the 32 lanes in
//     512-byte instructions; rows 8..15 land 64 bytes after rows 0..7, which
//     puts the rows the lanes read together on all 32 banks.  The block ids
//     of a warp's pages are held 32 at a time across its lanes.
//   * Integer codes enter the tensor cores without an arithmetic conversion:
//     one logic instruction per register moves two codes, offset to unsigned
//     (INT8 c + 128, INT4 c + 8), into the mantissa of two fp16 subnormals,
//     which are exactly (c + offset) * 2^-24; mma.sync m16n8k16 (fp16 in,
//     fp32 accumulate) then sums exact products.  The offset comes back out
//     once per dot product for K (offset * sum of the query) and once per
//     output for V (offset * sum of the PV operand, which one more MMA with
//     an all-ones A operand accumulates alongside O).  FP8 E4M3 codes are
//     converted by cvt.rn.f16x2.e4m3x2 (exact, no offset).  QK^T puts the 16
//     tokens of a page on M and the G <= 8 query heads on N; PV puts 16
//     head-dim rows on M and the query heads on N, with P transposed in
//     registers by movmatrix.  The head-dim order inside a lane is permuted
//     consistently for Q and K (a dot product does not depend on it).
//   * Pages whose 16 slots are all valid (all but a sequence's last) take a
//     path without per-slot masks.
//   * The per-token scales stay out of the inner products: logit =
//     (q' . c) * scale_k * (sm_scale * log2 e * 2^-e_q), and the PV operand is
//     p * scale_v * 2^-E.  q' = q * 2^e_q and the warp-wide power of two 2^-E
//     keep both fp16 operands in range without rounding q.
//   * Online softmax per warp in the log2 domain with a lazy rescale (the
//     running max moves only when a page exceeds it by 4), then a CTA-level
//     merge of the warps; the split partials (m, l, o) go to the workspace and
//     a second kernel merges the splits and the sinks.
//   * With H2O on, the split kernel writes each slot's fp32 logits; the merge
//     kernel, once the global (max, sum) of every query head is known, adds
//     sum_g exp2(logit - M_g) / L_g to every slot's score.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "kvc_device.h"
#include "kvc_internal.h"
#include "kvc_mma.h"

namespace kvc {
namespace {

using namespace dev;
using namespace codes;

constexpr int kWarps = 4;
constexpr int kPagesPerIter = 2;     // pages of a warp processed together in the split kernel
constexpr float kLazy = 4.0f;        // log2 units the running max may lag
constexpr int kMergeBtStage = 2048;  // block-table entries staged in shared memory (32768 slots)
constexpr int kMergeThreads = 512;

// One stage of a warp's ring holds one head-page: its K code rows, its V code
// rows, 16 K scales and 16 V scales (a K or V head-page is one contiguous run
// of 16 rows in the pool).  The 16-byte chunks of the code rows are placed by
// a fixed permutation (chunk_off) chosen so that every copy instruction and
// every read instruction of the kernel touches each shared-memory bank at most
// once per 128 bytes: chunk j of row t goes to
//   INT4 (4 chunks a row): 16 (8 (t >> 1) + 4 ((t ^ t >> 1 ^ t >> 2) & 1) + ((j + 2 (t >> 3)) & 3)),
//   8-bit (8 chunks a row): 128 t + 16 (j ^ (2 ((t >> 2) & 3) ^ 4 ((t >> 1) & 1))).
template <int BITS>
struct Geom {
  static constexpr int kRowBytes = BITS * 16;            // 128 (8-bit codes) or 64 (INT4)
  static constexpr int kK = 0;
  static constexpr int kV = 16 * kRowBytes;
  static constexpr int kKS = 32 * kRowBytes;
  static constexpr int kVS = kKS + 64;
  static constexpr int kStage = kVS + 64;
  static constexpr int kStages = 4;
  static constexpr int kSmem = kWarps * kStages * kStage;
  static constexpr int kChunksPerRow = kRowBytes / 16;
  static constexpr int kCopies = 16 * kRowBytes / 512;   // 16-byte copies per lane per K (or V) run
  static __host__ __device__ constexpr int chunk_off(int t, int j) {
    return BITS == 4 ? 16 * (8 * (t >> 1) + 4 * ((t ^ (t >> 1) ^ (t >> 2)) & 1) + ((j + 2 * (t >> 3)) & 3))
                     : 128 * t + 16 * (j ^ ((2 * ((t >> 2) & 3)) ^ (4 * ((t >> 1) & 1))));
  }
};

// The code rows of one page of one head into a stage, when `pred`: lane L
// copies the 16-byte chunks L + 32 i of the K run and of the V run (every
// instruction reads 512 contiguous bytes) to their permuted places d[i]
// (V: + kV).
template <int BITS>
__device__ __forceinline__ void copy_codes(bool pred, uint32_t sb, const uint32_t (&d)[Geom<BITS>::kCopies],
                                           const uint8_t* gK, const uint8_t* gV, uint64_t pol) {
  constexpr int kV = Geom<BITS>::kV;
  if (BITS == 8) {
    asm volatile(
        "{\n .reg .pred q;\n setp.ne.u32 q, %7, 0;\n"
        " @q cp.async.cg.shared.global.L2::cache_hint [%0], [%4], 16, %8;\n"
        " @q cp.async.cg.shared.global.L2::cache_hint [%1], [%4+512], 16, %8;\n"
        " @q cp.async.cg.shared.global.L2::cache_hint [%2], [%4+1024], 16, %8;\n"
        " @q cp.async.cg.shared.global.L2::cache_hint [%3], [%4+1536], 16, %8;\n"
        " @q cp.async.cg.shared.global.L2::cache_hint [%0+%6], [%5], 16, %8;\n"
        " @q cp.async.cg.shared.global.L2::cache_hint [%1+%6], [%5+512], 16, %8;\n"
        " @q cp.async.cg.shared.global.L2::cache_hint [%2+%6], [%5+1024], 16, %8;\n"
        " @q cp.async.cg.shared.global.L2::cache_hint [%3+%6], [%5+1536], 16, %8;\n}\n" ::"r"(sb + d[0]),
        "r"(sb + d[1 % Geom<BITS>::kCopies]), "r"(sb + d[2 % Geom<BITS>::kCopies]),
        "r"(sb + d[3 % Geom<BITS>::kCopies]), "l"(gK), "l"(gV), "n"(kV), "r"((uint32_t)pred), "l"(pol));
  } else {
    asm volatile(
        "{\n .reg .pred q;\n setp.ne.u32 q, %5, 0;\n"
        " @q cp.async.cg.shared.global.L2::cache_hint [%0], [%2], 16, %6;\n"
        " @q cp.async.cg.shared.global.L2::cache_hint [%1], [%2+512], 16, %6;\n"
        " @q cp.async.cg.shared.global.L2::cache_hint [%0+%4], [%3], 16, %6;\n"
        " @q cp.async.cg.shared.global.L2::cache_hint [%1+%4], [%3+512], 16, %6;\n}\n" ::"r"(sb + d[0]),
        "r"(sb + d[1]), "l"(gK), "l"(gV), "n"(kV), "r"((uint32_t)pred), "l"(pol));
  }
}

// FP8: the 8-bit codes are FP8 E4M3 instead of INT8 (same layout, same
// scales; only the code -> fp16 conversion differs, and no offset).
template <int BITS, bool FP8 = false>
__global__ void __launch_bounds__(kWarps * 32) attn_split_kernel(DevState s, int seq_begin, int batch,
                                                                 const uint16_t* __restrict__ q,
                                                                 float qk_scale_log2, AttnWork w,
                                                                 int spill) {
  using Gm = Geom<BITS>;
  constexpr int STAGES = Gm::kStages;
  constexpr int RB = Gm::kRowBytes;
  static_assert((STAGES & (STAGES - 1)) == 0, "ring positions are page index & (STAGES - 1)");
  constexpr bool kOffset = !FP8;  // integer codes as offset subnormals
  // the code offset times 2^-24 (K: subtracted from each dot product in units
  // of the query's sum) and the scale that brings the subnormal sums back
  constexpr float kOffK = BITS == 8 ? 128.0f * 0x1p-24f : 8.0f * 0x1p-24f;
  constexpr float kOffV = BITS == 8 ? 128.0f : 8.0f;
  __shared__ int cum[kMaxCallBatch + 1];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  pages_prefix(s, seq_begin, batch, cum);
  if (blockIdx.x == 0) {
    // the page prefix and zeroed tickets for the kernel that follows the split
    for (int i = threadIdx.x; i <= batch; i += blockDim.x) {
      w.cum[i] = cum[i];
      if (i < batch) w.seq_ticket[i] = 0;
    }
  }

  const int G = s.group;
  const int hkv = s.hkv;
  const int r = lane >> 2;
  const int c = lane & 3;
  const long long T = (long long)hkv * cum[batch];
  const int N = gridDim.x;
  const int cta = blockIdx.x;
  long long F = (long long)cta * T / N;
  const long long F1 = (long long)(cta + 1) * T / N;

  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t ring_s = smem_u32(smem) + warp * STAGES * Gm::kStage;
  const uint8_t* ring = smem + warp * STAGES * Gm::kStage;

  // what this lane copies of a page: chunks lane + 32 i of the K and V runs,
  // and (lanes 0..7) one 16-byte chunk of the 16 K or 16 V scales
  uint32_t cp_d[Gm::kCopies];
#pragma unroll
  for (int i = 0; i < Gm::kCopies; ++i)
    cp_d[i] = Gm::chunk_off((lane + 32 * i) / Gm::kChunksPerRow, (lane + 32 * i) % Gm::kChunksPerRow);
  const uint32_t sc_soff = lane < 4 ? Gm::kKS + 16 * lane : Gm::kVS + 16 * (lane - 4);
  // (lanes 8..31 get an address inside the scales too, never used)
  const float* sc_gbase = (lane < 4 ? s.k_scale : s.v_scale) + 4 * (lane & 3);
  // what this lane reads of a stage: the chunks of K rows 2r and 2r+1 holding
  // dims 32c.. (INT4) or 16c.. and 64+16c.. (8-bit); of V rows 4c..4c+3 the
  // 8 bytes at 8r (INT4) or 16 bytes at 16r; the scales of slots 2r and 2r+1
  int k_off[BITS == 8 ? 4 : 2], v_off[4];
  if (BITS == 8) {
    k_off[0] = Gm::chunk_off(2 * r, c);
    k_off[1] = Gm::chunk_off(2 * r, c + 4);
    k_off[2] = Gm::chunk_off(2 * r + 1, c);
    k_off[3 % (BITS == 8 ? 4 : 2)] = Gm::chunk_off(2 * r + 1, c + 4);
  } else {
    k_off[0] = Gm::chunk_off(2 * r, c);
    k_off[1] = Gm::chunk_off(2 * r + 1, c);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k)
    v_off[k] = Gm::kV + (BITS == 8 ? Gm::chunk_off(4 * c + k, r) : Gm::chunk_off(4 * c + k, r >> 1) + 8 * (r & 1));
  const int s_off = Gm::kKS + 8 * r;
  // L2 policies: the KV stream is read once (evict first); the logit spill is
  // read back by the next kernel (evict last)
  const uint64_t kv_pol = l2_evict_first();
  const uint64_t spill_pol = l2_evict_last();

  while (F < F1) {
    // ---- the (sequence, KV head) pair of page F and this CTA's run of its pages
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((long long)hkv * cum[mid] <= F) lo = mid; else hi = mid - 1;
    }
    const int bl = lo;
    const int b = seq_begin + bl;
    const int npg = cum[bl + 1] - cum[bl];
    const long long pbase = (long long)hkv * cum[bl];
    const int h = (int)((F - pbase) / npg);
    const long long Pf = pbase + (long long)h * npg;
    const int pg_a = (int)(F - Pf);
    const int pg_e = (int)((F1 < Pf + npg ? F1 : Pf + npg) - Pf);
    const int S = s.seq_slots[b];
    const int pair = bl * hkv + h;

    // ---- page pipeline: this warp takes pages pg_a + warp, + kWarps, ...
    const int n_range = pg_e - pg_a;
    const int n_my = n_range > warp ? (n_range - warp + kWarps - 1) / kWarps : 0;
    const int32_t* bt = s.block_table + (size_t)b * s.max_bps;
    // block ids of this warp's pages, 32 at a time across the lanes (the
    // next 32 loaded while the current ones are used)
    auto bt_load = [&](int chunk) -> int {
      const int kk = chunk * 32 + lane;
      return kk < n_my ? bt[pg_a + warp + kWarps * kk] : -1;
    };
    int bt_cur = bt_load(0);
    int bt_nxt = n_my > 32 ? bt_load(1) : -1;
    uint32_t stage_ok = 0;  // bit k: the page in stage k has a valid block id
    // this lane's source bases for head h (a block's head-page = base + block x stride)
    const uint8_t* kb = s.k_codes + (size_t)h * (16 * RB) + 16 * lane;
    const uint8_t* vb = s.v_codes + (size_t)h * (16 * RB) + 16 * lane;
    const float* scb = sc_gbase + (size_t)h * kPage;
    const uint32_t code_stride = (uint32_t)hkv * (16 * RB), sc_stride = (uint32_t)hkv * kPage;

    // page k of this warp into stage k & (STAGES - 1), one commit group (empty
    // past n_my: the block ids there are -1)
    auto issue = [&](int k) {
      if ((k & 31) == 0 && k > 0) {
        bt_cur = bt_nxt;
        bt_nxt = bt_load((k >> 5) + 1);
      }
      const int blk = __shfl_sync(0xffffffffu, bt_cur, k & 31);
      const bool ok = (unsigned)blk < (unsigned)s.num_blocks;
      const int slot_issue = k & (STAGES - 1);
      stage_ok = (stage_ok & ~(1u << slot_issue)) | ((uint32_t)ok << slot_issue);
      const uint32_t sb = ring_s + slot_issue * Gm::kStage;
      const size_t off = (size_t)(uint32_t)blk * code_stride;
      copy_codes<BITS>(ok, sb, cp_d, kb + off, vb + off, kv_pol);
      cp_async16_if(ok && lane < 8, sb + sc_soff, scb + (size_t)(uint32_t)blk * sc_stride);
      cp_async_commit();
    };

    // pages [0, nxt) are issued, one commit group each (empty past n_my)
    int nxt = 0;
    auto issue_upto = [&](int n) {
#pragma unroll 1
      for (; nxt < n; ++nxt) issue(nxt);
    };
    issue_upto(kPagesPerIter == 2 ? 2 : STAGES - 1);

    // ---- query fragments (B operand of QK^T), scaled by 2^e_g into fp16 range;
    // with offset codes, the sum of each head's query values as the MMA sees them
    uint32_t bq[8][2];
    float cq0, cq1, ch0 = 0.0f, ch1 = 0.0f;
    {
      float qv[32];
      const int g = r;
      if (g < G) {
        // the lane's 32 dims, in the order of its K codes: 8-bit dims
        // 16c..16c+15 and 64+16c..64+16c+15, INT4 dims 32c..32c+31
        const uint16_t* qrow = q + ((size_t)bl * s.hq + h * G + g) * kHeadDim;
        const uint4* src_a = reinterpret_cast<const uint4*>(qrow + (BITS == 8 ? 16 * c : 32 * c));
        const uint4* src_b = reinterpret_cast<const uint4*>(qrow + (BITS == 8 ? 64 + 16 * c : 32 * c + 16));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 u = i < 2 ? src_a[i] : src_b[i - 2];
          const uint32_t ws[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            qv[8 * i + 2 * j] = bf16f(ws[j] & 0xFFFFu);
            qv[8 * i + 2 * j + 1] = bf16f(ws[j] >> 16);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) qv[i] = 0.0f;
      }
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(qv[i]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      int e = 0;
      if (amax > 0.0f) e = min(max(14 - exponent_of(amax), -100), 100);
      const float f2e = pow2i(e);  // multiplying by a power of two is exact here
#pragma unroll
      for (int i = 0; i < 32; ++i) qv[i] *= f2e;
      // the B fragment pairs each A register's two codes: 8-bit offset codes
      // give (b0, b2) and (b1, b3) of a word, E4M3 (b0, b1) and (b2, b3); INT4
      // gives the low nibbles of bytes 0 and 2, then their high nibbles (16x:
      // the query's matching values are divided by 16, exactly)
      if (BITS == 8) {
#pragma unroll
        for (int st = 0; st < 8; ++st) {
          if (FP8) {
            bq[st][0] = pack_half2(qv[4 * st + 0], qv[4 * st + 1]);
            bq[st][1] = pack_half2(qv[4 * st + 2], qv[4 * st + 3]);
          } else {
            bq[st][0] = pack_half2(qv[4 * st + 0], qv[4 * st + 2]);
            bq[st][1] = pack_half2(qv[4 * st + 1], qv[4 * st + 3]);
          }
        }
      } else {
        constexpr float k16 = 0.0625f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          bq[2 * i][0] = pack_half2(qv[8 * i + 0], qv[8 * i + 4]);
          bq[2 * i][1] = pack_half2(qv[8 * i + 1] * k16, qv[8 * i + 5] * k16);
          bq[2 * i + 1][0] = pack_half2(qv[8 * i + 2], qv[8 * i + 6]);
          bq[2 * i + 1][1] = pack_half2(qv[8 * i + 3] * k16, qv[8 * i + 7] * k16);
        }
      }
      if (kOffset) {
        // sum of q' over the head's 128 dims, from the fp16 values fed to the MMA
        float qs = 0.0f;
#pragma unroll
        for (int st = 0; st < 8; ++st) {
          const float2 a = unpack_half2(bq[st][0]);
          const float2 bb = unpack_half2(bq[st][1]);
          const float fb = BITS == 4 ? 16.0f : 1.0f;
          qs += (a.x + a.y) + fb * (bb.x + bb.y);
        }
        qs += __shfl_xor_sync(0xffffffffu, qs, 1);
        qs += __shfl_xor_sync(0xffffffffu, qs, 2);
        ch0 = kOffK * __shfl_sync(0xffffffffu, qs, (2 * c) * 4);
        ch1 = kOffK * __shfl_sync(0xffffffffu, qs, (2 * c + 1) * 4);
      }
      const int e0 = __shfl_sync(0xffffffffu, e, (2 * c) * 4);
      const int e1 = __shfl_sync(0xffffffffu, e, (2 * c + 1) * 4);
      // offset codes carry 2^-24: scale the dot products back by 2^24
      cq0 = qk_scale_log2 * pow2i((kOffset ? 24 : 0) - e0);
      cq1 = qk_scale_log2 * pow2i((kOffset ? 24 : 0) - e1);
    }

    float oacc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.0f;
    float osum[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // offset codes: sum over slots of the PV operand
    float m0 = kNegBig, m1 = kNegBig, l0 = 0.0f, l1 = 0.0f;
    int E = 0;
    bool e_set = false;
    float sv_hi = 0.0f;
    float inv2E = 1.0f;
    // logits of this pair, [g][slot]; the lane writes slots (2r, 2r+1) of heads
    // 2c and 2c+1 (lanes of padding heads write nothing)
    const bool sp0 = spill && 2 * c < G, sp1 = spill && 2 * c + 1 < G;
    float* lg0p = w.logits + ((size_t)pair * G + (sp0 ? 2 * c : 0)) * w.s_cap + 2 * r;
    float* lg1p = w.logits + ((size_t)pair * G + (sp1 ? 2 * c + 1 : 0)) * w.s_cap + 2 * r;

    // NP consecutive pages of this warp (k .. k + NP - 1), their instructions
    // interleaved; FULL: every slot valid (the common case), no per-slot masks
    auto pages_body = [&](auto np_tag, auto full_tag, int k) {
      constexpr int NP = decltype(np_tag)::value;
      constexpr bool FULL = decltype(full_tag)::value;
      const uint8_t* st[NP];
      int slot0[NP];
      bool v0[NP], v1[NP];
      float2 skv[NP], svv[NP];
#pragma unroll
      for (int pp = 0; pp < NP; ++pp) {
        const int sc = (k + pp) & (STAGES - 1);
        const bool blk_ok = (stage_ok >> sc) & 1u;
        st[pp] = ring + sc * Gm::kStage;
        slot0[pp] = (pg_a + warp + kWarps * (k + pp)) * kPage;
        v0[pp] = FULL || (blk_ok && (slot0[pp] + 2 * r < S));
        v1[pp] = FULL || (blk_ok && (slot0[pp] + 2 * r + 1 < S));
        skv[pp] = *reinterpret_cast<const float2*>(st[pp] + s_off);
        svv[pp] = *reinterpret_cast<const float2*>(st[pp] + s_off + 64);
      }

      // ---- S = K_codes . q'  (rows: slots 2r and 2r+1, cols: query heads 2c, 2c+1)
      // the accumulators start at -(code offset x query sum), so they end at
      // the dot products of the query with the signed codes
      float acc[NP][4];
#pragma unroll
      for (int pp = 0; pp < NP; ++pp) {
        acc[pp][0] = acc[pp][2] = -ch0;
        acc[pp][1] = acc[pp][3] = -ch1;
      }
      if (BITS == 8) {
        uint32_t w0[NP][8], w1[NP][8];
#pragma unroll
        for (int pp = 0; pp < NP; ++pp) {
          const uint4 ka = *reinterpret_cast<const uint4*>(st[pp] + k_off[0]);
          const uint4 kb2 = *reinterpret_cast<const uint4*>(st[pp] + k_off[1]);
          const uint4 kc = *reinterpret_cast<const uint4*>(st[pp] + k_off[2 % (BITS == 8 ? 4 : 2)]);
          const uint4 kd = *reinterpret_cast<const uint4*>(st[pp] + k_off[3 % (BITS == 8 ? 4 : 2)]);
          w0[pp][0] = ka.x; w0[pp][1] = ka.y; w0[pp][2] = ka.z; w0[pp][3] = ka.w;
          w0[pp][4] = kb2.x; w0[pp][5] = kb2.y; w0[pp][6] = kb2.z; w0[pp][7] = kb2.w;
          w1[pp][0] = kc.x; w1[pp][1] = kc.y; w1[pp][2] = kc.z; w1[pp][3] = kc.w;
          w1[pp][4] = kd.x; w1[pp][5] = kd.y; w1[pp][6] = kd.z; w1[pp][7] = kd.w;
        }
#pragma unroll
        for (int stp = 0; stp < 8; ++stp) {
#pragma unroll
          for (int pp = 0; pp < NP; ++pp) {
            uint32_t a0, a1, a2, a3;
            if (FP8) {
              e4m3x4_to_h2(w0[pp][stp], a0, a2);
              e4m3x4_to_h2(w1[pp][stp], a1, a3);
            } else {
              a0 = u8_even(w0[pp][stp]);
              a1 = u8_even(w1[pp][stp]);
              a2 = u8_even(w0[pp][stp] >> 8);
              a3 = u8_even(w1[pp][stp] >> 8);
            }
            mma16816(acc[pp], a0, a1, a2, a3, bq[stp][0], bq[stp][1]);
          }
        }
      } else {
        uint32_t w0[NP][4], w1[NP][4];
#pragma unroll
        for (int pp = 0; pp < NP; ++pp) {
          const uint4 ka = *reinterpret_cast<const uint4*>(st[pp] + k_off[0]);
          const uint4 kb2 = *reinterpret_cast<const uint4*>(st[pp] + k_off[1]);
          w0[pp][0] = ka.x; w0[pp][1] = ka.y; w0[pp][2] = ka.z; w0[pp][3] = ka.w;
          w1[pp][0] = kb2.x; w1[pp][1] = kb2.y; w1[pp][2] = kb2.z; w1[pp][3] = kb2.w;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
          for (int pp = 0; pp < NP; ++pp) {
            const uint32_t x0 = w0[pp][i], x1 = w1[pp][i];
            const uint32_t x0s = x0 >> 8, x1s = x1 >> 8;
            mma16816(acc[pp], u4_lo(x0), u4_lo(x1), u4_hi(x0), u4_hi(x1), bq[2 * i][0], bq[2 * i][1]);
            mma16816(acc[pp], u4_lo(x0s), u4_lo(x1s), u4_hi(x0s), u4_hi(x1s), bq[2 * i + 1][0],
                     bq[2 * i + 1][1]);
          }
        }
      }
      float lg[NP][4];
#pragma unroll
      for (int pp = 0; pp < NP; ++pp) {
        lg[pp][0] = v0[pp] ? acc[pp][0] * (skv[pp].x * cq0) : -INFINITY;  // slot 2r,   head 2c
        lg[pp][1] = v0[pp] ? acc[pp][1] * (skv[pp].x * cq1) : -INFINITY;  // slot 2r,   head 2c+1
        lg[pp][2] = v1[pp] ? acc[pp][2] * (skv[pp].y * cq0) : -INFINITY;  // slot 2r+1, head 2c
        lg[pp][3] = v1[pp] ? acc[pp][3] * (skv[pp].y * cq1) : -INFINITY;  // slot 2r+1, head 2c+1
        st2_if_hint(sp0, lg0p + slot0[pp], lg[pp][0], lg[pp][2], spill_pol);
        st2_if_hint(sp1, lg1p + slot0[pp], lg[pp][1], lg[pp][3], spill_pol);
      }

      // ---- lazy online softmax: reduce and rescale only when some lane's
      // logit exceeds the running max by kLazy, or a V scale outgrows 2^(E+4)
      float tm0 = -INFINITY, tm1 = -INFINITY, svl = 0.0f;
#pragma unroll
      for (int pp = 0; pp < NP; ++pp) {
        tm0 = fmaxf(tm0, fmaxf(lg[pp][0], lg[pp][2]));
        tm1 = fmaxf(tm1, fmaxf(lg[pp][1], lg[pp][3]));
        svl = fmaxf(svl, fmaxf(v0[pp] ? svv[pp].x : 0.0f, v1[pp] ? svv[pp].y : 0.0f));
      }
      const bool need = tm0 > m0 + kLazy || tm1 > m1 + kLazy || svl > sv_hi || (!e_set && svl > 0.0f);
      if (__any_sync(0xffffffffu, need)) {
        float svm = svl;
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          tm0 = fmaxf(tm0, __shfl_xor_sync(0xffffffffu, tm0, o));
          tm1 = fmaxf(tm1, __shfl_xor_sync(0xffffffffu, tm1, o));
          svm = fmaxf(svm, __shfl_xor_sync(0xffffffffu, svm, o));
        }
        const float nm0 = fmaxf(m0, tm0), nm1 = fmaxf(m1, tm1);
        const float al0 = fast_exp2(m0 - nm0), al1 = fast_exp2(m1 - nm1);
        const bool rescale_e = svm > sv_hi || (!e_set && svm > 0.0f);
        int nE = E;
        if (rescale_e) nE = min(max(exponent_of(svm), -126), 126);
        const int dE = E - nE;  // <= 0 once E is set; up to +126 on the first page (O is 0 then)
        const float f = dE >= -126 ? pow2i(min(dE, 127)) : 0.0f;
        const float f0 = al0 * f, f1 = al1 * f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          oacc[j][0] *= f0;
          oacc[j][2] *= f0;
          oacc[j][1] *= f1;
          oacc[j][3] *= f1;
        }
        osum[0] *= f0;
        osum[2] *= f0;
        osum[1] *= f1;
        osum[3] *= f1;
        l0 *= al0;
        l1 *= al1;
        m0 = nm0;
        m1 = nm1;
        if (rescale_e) {
          E = nE;
          e_set = true;
          sv_hi = pow2i(min(E + 4, 127));
          inv2E = pow2i(-E);
        }
      }
      uint32_t pb0[NP], pb1[NP];
#pragma unroll
      for (int pp = 0; pp < NP; ++pp) {
        const float sn0 = v0[pp] ? svv[pp].x * inv2E : 0.0f;
        const float sn1 = v1[pp] ? svv[pp].y * inv2E : 0.0f;
        const float p0 = fast_exp2(lg[pp][0] - m0), p1 = fast_exp2(lg[pp][1] - m1);
        const float p2 = fast_exp2(lg[pp][2] - m0), p3 = fast_exp2(lg[pp][3] - m1);
        l0 += p0 + p2;
        l1 += p1 + p3;
        pb0[pp] = movmatrix_t(pack_half2(p0 * sn0, p1 * sn0));
        pb1[pp] = movmatrix_t(pack_half2(p2 * sn1, p3 * sn1));
      }

      // ---- O^T += V_codes^T . P~^T   (rows: head-dim 16r + 2j (+1), cols: query heads)
#pragma unroll
      for (int pp = 0; pp < NP; ++pp) {
        if (BITS == 8) {
          const uint4 r0 = *reinterpret_cast<const uint4*>(st[pp] + v_off[0]);
          const uint4 r1 = *reinterpret_cast<const uint4*>(st[pp] + v_off[1]);
          const uint4 r2 = *reinterpret_cast<const uint4*>(st[pp] + v_off[2]);
          const uint4 r3 = *reinterpret_cast<const uint4*>(st[pp] + v_off[3]);
          const uint32_t x0[4] = {r0.x, r0.y, r0.z, r0.w};  // slot 4c
          const uint32_t x1[4] = {r1.x, r1.y, r1.z, r1.w};  // slot 4c+1
          const uint32_t x2[4] = {r2.x, r2.y, r2.z, r2.w};  // slot 4c+2
          const uint32_t x3[4] = {r3.x, r3.y, r3.z, r3.w};  // slot 4c+3
#pragma unroll
          for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const int j = 2 * wd + half;
              // byte k of x and of y in bytes 0 and 2: pairs slots (4c, 4c+2) or (4c+1, 4c+3)
              const uint32_t sa = (2 * half) | ((4 + 2 * half) << 8);
              const uint32_t sb = (2 * half + 1) | ((5 + 2 * half) << 8);
              uint32_t a0, a1, a2, a3;
              if (FP8) {
                a0 = e4m3_pair_to_h2(x0[wd], x2[wd], 2 * half);
                a1 = e4m3_pair_to_h2(x0[wd], x2[wd], 2 * half + 1);
                a2 = e4m3_pair_to_h2(x1[wd], x3[wd], 2 * half);
                a3 = e4m3_pair_to_h2(x1[wd], x3[wd], 2 * half + 1);
              } else {
                a0 = u8_even(prmt(x0[wd], x2[wd], sa));
                a1 = u8_even(prmt(x0[wd], x2[wd], sb));
                a2 = u8_even(prmt(x1[wd], x3[wd], sa));
                a3 = u8_even(prmt(x1[wd], x3[wd], sb));
              }
              mma16816(oacc[j], a0, a1, a2, a3, pb0[pp], pb1[pp]);
            }
          }
        } else {
          const uint2 r0 = *reinterpret_cast<const uint2*>(st[pp] + v_off[0]);
          const uint2 r1 = *reinterpret_cast<const uint2*>(st[pp] + v_off[1]);
          const uint2 r2 = *reinterpret_cast<const uint2*>(st[pp] + v_off[2]);
          const uint2 r3 = *reinterpret_cast<const uint2*>(st[pp] + v_off[3]);
          const uint32_t x0[2] = {r0.x, r0.y};
          const uint32_t x1[2] = {r1.x, r1.y};
          const uint32_t x2[2] = {r2.x, r2.y};
          const uint32_t x3[2] = {r3.x, r3.y};
#pragma unroll
          for (int u = 0; u < 2; ++u) {
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              // bytes 2m, 2m+1 of slots (4c, 4c+2) and of (4c+1, 4c+3), one pair per 16-bit half
              const uint32_t sel = m == 0 ? 0x5410u : 0x7632u;
              const uint32_t v02 = prmt(x0[u], x2[u], sel);
              const uint32_t v13 = prmt(x1[u], x3[u], sel);
              const uint32_t v02s = v02 >> 8, v13s = v13 >> 8;
              mma16816(oacc[4 * u + 2 * m], u4_lo(v02), u4_hi(v02), u4_lo(v13), u4_hi(v13), pb0[pp], pb1[pp]);
              mma16816(oacc[4 * u + 2 * m + 1], u4_lo(v02s), u4_hi(v02s), u4_lo(v13s), u4_hi(v13s), pb0[pp],
                       pb1[pp]);
            }
          }
        }
        if (kOffset) {
          constexpr uint32_t kOne = 0x3C003C00u;  // fp16 (1, 1)
          mma16816(osum, kOne, kOne, kOne, kOne, pb0[pp], pb1[pp]);
        }
      }
    };
    // this warp's pages k < k_full have all 16 slots below S
    const int full_pages = S / kPage;
    const int k_full = full_pages > pg_a + warp ? min(n_my, (full_pages - pg_a - warp + kWarps - 1) / kWarps) : 0;
    int k = 0;
    if (kPagesPerIter == 2) {
      // two full pages per iteration, the copies of the next two in flight;
      // on entry pages [0, k + 2) are issued
#pragma unroll 1
      for (; k + 1 < k_full; k += 2) {
        if (((stage_ok >> (k & (STAGES - 1))) & 3u) != 3u) break;  // a bad block id: the slow path
        issue(k + 2);
        issue(k + 3);
        nxt = k + 4;
        cp_async_wait<2>();
        __syncwarp();
        pages_body(std::integral_constant<int, 2>{}, std::true_type{}, k);
        __syncwarp();
      }
    }
    // one page at a time: the pages through k + STAGES - 1 issued (into the
    // stages of pages already consumed), page k waited for
#pragma unroll 1
    for (; k < n_my; ++k) {
      issue_upto(k + STAGES);
      cp_async_wait<STAGES - 1>();
      __syncwarp();
      const bool ok = (stage_ok >> (k & (STAGES - 1))) & 1u;
      if (!ok && lane == 0) atomicOr(&s.counters[kCtrStatus], kDevBadBlockId);
      if (ok && k < k_full)
        pages_body(std::integral_constant<int, 1>{}, std::true_type{}, k);
      else
        pages_body(std::integral_constant<int, 1>{}, std::false_type{}, k);
      __syncwarp();
    }
    cp_async_wait<0>();

    // ---- per-warp totals, CTA merge of the 4 warps, partial to the workspace
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    const float f2E = pow2i(E);
    __syncthreads();  // every warp is done with its ring: reuse shared memory
    float* sm_m = reinterpret_cast<float*>(smem);  // [kWarps][8]
    float* sm_l = sm_m + kWarps * kMaxGroup;       // [kWarps][8]
    float* sm_o = sm_l + kWarps * kMaxGroup;       // [kWarps][8][128]
    if (r == 0) {
      sm_m[warp * kMaxGroup + 2 * c] = m0;
      sm_m[warp * kMaxGroup + 2 * c + 1] = m1;
      sm_l[warp * kMaxGroup + 2 * c] = l0;
      sm_l[warp * kMaxGroup + 2 * c + 1] = l1;
    }
    {
      // offset codes: o = (2^24 acc - offset x sum of the PV operand) 2^E,
      // with 2^20 for the rows of INT4 high nibbles (16x)
      const float sA = kOffset ? 0x1p24f : 1.0f;
      const float sB = kOffset ? (BITS == 4 ? 0x1p20f : 0x1p24f) : 1.0f;
      const float b0 = kOffset ? kOffV * osum[0] : 0.0f;
      const float b1 = kOffset ? kOffV * osum[1] : 0.0f;
      float* o0 = sm_o + ((size_t)warp * kMaxGroup + 2 * c) * kHeadDim + 16 * r;
      float* o1 = o0 + kHeadDim;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        o0[2 * j] = (oacc[j][0] * sA - b0) * f2E;
        o0[2 * j + 1] = (oacc[j][2] * sB - b0) * f2E;
        o1[2 * j] = (oacc[j][1] * sA - b1) * f2E;
        o1[2 * j + 1] = (oacc[j][3] * sB - b1) * f2E;
      }
    }
    __syncthreads();
    const int d = threadIdx.x;  // 128 threads = head_dim
    const size_t pslot = (size_t)pair + cta;
    for (int g = 0; g < G; ++g) {
      float M = kNegBig;
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww) M = fmaxf(M, sm_m[ww * kMaxGroup + g]);
      float o = 0.0f, l = 0.0f;
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww) {
        const float wt = fast_exp2(sm_m[ww * kMaxGroup + g] - M);
        o += wt * sm_o[((size_t)ww * kMaxGroup + g) * kHeadDim + d];
        l += wt * sm_l[ww * kMaxGroup + g];
      }
      w.part_o[(pslot * G + g) * kHeadDim + d] = o;
      if (d == 0) {
        w.part_ml[(pslot * G + g) * 2 + 0] = M;
        w.part_ml[(pslot * G + g) * 2 + 1] = l;
      }
    }
    __syncthreads();  // shared memory is reused by the next pair
    F = Pf + pg_e;
  }
}

// Merge the stream-K partials and the bf16 sinks of one (sequence, KV head);
// write the bf16 outputs of its G query heads and their (M, L) to w.stats;
// add this step's probabilities to the sink scores (kMergeSinkScores) and
// also to the bf16 window's and every pool slot's scores (kMergeAllScores).
__global__ void __launch_bounds__(kMergeThreads, 2) attn_merge_kernel(DevState s, int seq_begin, int batch,
                                                                     const uint16_t* __restrict__ q,
                                                                     uint16_t* __restrict__ out,
                                                                     float qk_scale_log2, AttnWork w, int accumulate) {
  __shared__ MergeShared ms;
  __shared__ int32_t sh_bt[kMergeBtStage];
  const int h = blockIdx.x;
  const int bl = blockIdx.y;
  // the page prefix of the slice, as the split kernel's first CTA published it
  merge_phase(s, seq_begin, batch, w.cum, h, bl, q, out, qk_scale_log2, w, accumulate != kMergeNoScores, ms);
  if (accumulate != kMergeAllScores) return;
  ring_score_pass(s, w, seq_begin + bl, bl, h, ms);
  // score pass: the sequence's block-table row is staged in shared memory
  // (when it fits) and each thread handles 4 slots with all loads issued first
  const int b = seq_begin + bl;
  const int G = s.group;
  const int hkv = s.hkv;
  const int S = s.seq_slots[b];
  const int pair = bl * hkv + h;
  const int32_t* bt = s.block_table + (size_t)b * s.max_bps;
  const int npages = (S + kPage - 1) / kPage;
  const int32_t* btp = bt;
  if (npages <= kMergeBtStage) {
    for (int i = threadIdx.x; i < npages; i += blockDim.x) sh_bt[i] = bt[i];
    btp = sh_bt;
  }
  __syncthreads();
  const float* lgr = w.logits + (size_t)pair * G * w.s_cap;
  const int nt = blockDim.x;
  for (int t0 = threadIdx.x; t0 < S; t0 += 4 * nt) {
    int blk[4];
    float inc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = t0 + u * nt;
      blk[u] = t < S ? btp[t / kPage] : -1;
      inc[u] = t < S ? h2o_increment(lgr, w.s_cap, t, G, ms) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = t0 + u * nt;
      if (t < S && (unsigned)blk[u] < (unsigned)s.num_blocks)
        s.score[((size_t)blk[u] * hkv + h) * kPage + (t % kPage)] += inc[u];
    }
  }
}

// cudaFuncSetAttribute is per device and per kernel: one flag per (BITS, device).
template <int BITS, bool FP8 = false>
cudaError_t ensure_split_smem() {
  static int done[64] = {0};
  return opt_in_smem(reinterpret_cast<const void*>(attn_split_kernel<BITS, FP8>), Geom<BITS>::kSmem, done);
}

template <int BITS, bool FP8 = false>
int split_ctas_per_sm() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  if (ensure_split_smem<BITS, FP8>() != cudaSuccess) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_split_kernel<BITS, FP8>, kWarps * 32,
                                                    Geom<BITS>::kSmem) !=
          cudaSuccess ||
      n < 1)
    n = 1;
  if (dev < 64) cached[dev] = n;
  return n;
}

}  // namespace

int attention_smem_bytes(int bits) { return bits == 8 ? Geom<8>::kSmem : Geom<4>::kSmem; }

int attention_ctas_per_sm(int bits, bool fp8) {
  if (bits == 8) return fp8 ? split_ctas_per_sm<8, true>() : split_ctas_per_sm<8>();
  return split_ctas_per_sm<4>();
}

template <int BITS, bool FP8>
cudaError_t launch_split_t(const DevState& s, int seq_begin, int batch, const uint16_t* q, float qk_scale_log2,
                           const AttnWork& w, bool spill, cudaStream_t st) {
  const cudaError_t e = ensure_split_smem<BITS, FP8>();
  if (e != cudaSuccess) return e;
  attn_split_kernel<BITS, FP8><<<w.ncta, kWarps * 32, Geom<BITS>::kSmem, st>>>(s, seq_begin, batch, q,
                                                                               qk_scale_log2, w, spill);
  return cudaGetLastError();
}

cudaError_t launch_attention_split(const DevState& s, int seq_begin, int batch, const uint16_t* q,
                                   float qk_scale_log2, const AttnWork& w, bool spill, cudaStream_t st) {
  if (s.bits == 8)
    return s.fp8 ? launch_split_t<8, true>(s, seq_begin, batch, q, qk_scale_log2, w, spill, st)
                 : launch_split_t<8, false>(s, seq_begin, batch, q, qk_scale_log2, w, spill, st);
  return launch_split_t<4, false>(s, seq_begin, batch, q, qk_scale_log2, w, spill, st);
}

cudaError_t launch_attention_merge(const DevState& s, int seq_begin, int batch, const uint16_t* q, uint16_t* out,
                                   float qk_scale_log2, const AttnWork& w, MergeScores scores, cudaStream_t st) {
  dim3 grid(s.hkv, batch);
  attn_merge_kernel<<<grid, kMergeThreads, 0, st>>>(s, seq_begin, batch, q, out, qk_scale_log2, w, (int)scores);
  return cudaGetLastError();
}

}  // namespace kvc
