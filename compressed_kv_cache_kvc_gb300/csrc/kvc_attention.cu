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
//     stages with cp.async (16-byte, coalesced: a K or V page of one head is
//     one contiguous 2 KB (INT8) / 1 KB (INT4) run of the pool).
//   * Codes are exact small integers, so they are converted to fp16 exactly
//     (byte-permute + magic-number subtraction, the integer-to-float trick of
//     Kim et al., "Who Says Elephants Can't Run", 2022) and fed straight from
//     registers to mma.sync m16n8k16 (fp16 in, fp32 accumulate).  QK^T puts the
//     16 tokens of a page on M and the G <= 8 query heads on N; PV puts 16
//     head-dim rows on M and the query heads on N, with P transposed in
//     registers by movmatrix.  The head-dim order inside a lane is permuted
//     consistently for Q and K (a dot product does not depend on it).
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

#include "kvc_device.h"
#include "kvc_internal.h"

namespace kvc {
namespace {

using namespace dev;

constexpr int kWarps = 4;
constexpr float kLazy = 4.0f;        // log2 units the running max may lag
constexpr int kMergeBtStage = 2048;  // block-table entries staged in shared memory (32768 slots)
constexpr int kMergeThreads = 512;

template <int BITS>
struct Geom {
  static constexpr int kRowBytes = BITS * 16;           // 128 (INT8) or 64 (INT4)
  static constexpr int kKBytes = BITS == 8 ? 2048 : 1024;
  static constexpr int kVBytes = BITS == 8 ? 2048 : 1024;
  static constexpr int kStage = kKBytes + kVBytes + 128;  // + 16 K scales + 16 V scales
  static constexpr int kStages = 4;  // INT8: 3 CTAs/SM by shared memory, INT4: 4
  static constexpr int kSmem = kWarps * kStages * kStage;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async16_s(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src));
}
// All code chunks of one page for this lane (see the lane offsets in the
// split kernel): K then V, at fixed immediate distances from the lane bases.
template <int BITS>
__device__ __forceinline__ void copy_page(uint32_t sK, const uint8_t* kg, uint32_t sV, const uint8_t* vg) {
  if (BITS == 8) {
    asm volatile(
        "cp.async.cg.shared.global [%0], [%1], 16;\n"
        "cp.async.cg.shared.global [%0+512], [%1+64], 16;\n"
        "cp.async.cg.shared.global [%0+1024], [%1+128], 16;\n"
        "cp.async.cg.shared.global [%0+1536], [%1+192], 16;\n"
        "cp.async.cg.shared.global [%2], [%3], 16;\n"
        "cp.async.cg.shared.global [%2+512], [%3+128], 16;\n"
        "cp.async.cg.shared.global [%2+1024], [%3+256], 16;\n"
        "cp.async.cg.shared.global [%2+1536], [%3+384], 16;\n" ::"r"(sK), "l"(kg), "r"(sV), "l"(vg));
  } else {
    asm volatile(
        "cp.async.cg.shared.global [%0], [%1], 16;\n"
        "cp.async.cg.shared.global [%0+512], [%1+64], 16;\n"
        "cp.async.ca.shared.global [%2], [%3], 8;\n"
        "cp.async.ca.shared.global [%2+256], [%3+64], 8;\n"
        "cp.async.ca.shared.global [%2+512], [%3+128], 8;\n"
        "cp.async.ca.shared.global [%2+768], [%3+192], 8;\n" ::"r"(sK), "l"(kg), "r"(sV), "l"(vg));
  }
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) { return __byte_perm(a, b, sel); }
__device__ __forceinline__ uint32_t as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) { return as_u32(__hsub2(as_h2(a), as_h2(b))); }
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  return as_u32(__hfma2(as_h2(a), as_h2(b), as_h2(c)));
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 4 INT8 codes (bytes b0..b3 of w, already XOR 0x80) -> fp16x2 (b0, b1) and (b2, b3).
__device__ __forceinline__ void i8x4_to_h2(uint32_t wx, uint32_t& lo, uint32_t& hi) {
  lo = hsub2(prmt(wx, 0x64646464u, 0x4140u), 0x64806480u);
  hi = hsub2(prmt(wx, 0x64646464u, 0x4342u), 0x64806480u);
}
// Byte k of x and byte k of y (INT8 codes) -> fp16x2 (x_k, y_k).
__device__ __forceinline__ uint32_t i8_pair_to_h2(uint32_t x, uint32_t y, uint32_t sel) {
  return hsub2((prmt(x, y, sel) & 0x00FF00FFu) ^ 0x64806480u, 0x64806480u);
}
// FP8 E4M3 codes -> fp16 (every E4M3 value is exact in fp16), by the
// conversion instruction: 4 codes (bytes b0..b3 of w) -> (b0, b1) and (b2, b3).
__device__ __forceinline__ void e4m3x4_to_h2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 l, h;\n"
      " mov.b32 {l, h}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, l;\n"
      " cvt.rn.f16x2.e4m3x2 %1, h;\n}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}
// Byte k of x and byte k of y (E4M3 codes) -> fp16x2 (x_k, y_k).
__device__ __forceinline__ uint32_t e4m3_pair_to_h2(uint32_t x, uint32_t y, int k) {
  const uint32_t pr = prmt(x, y, (uint32_t)k | ((uint32_t)(4 + k) << 4));
  uint32_t d;
  asm("{\n .reg .b16 l, h;\n"
      " mov.b32 {l, h}, %1;\n"
      " cvt.rn.f16x2.e4m3x2 %0, l;\n}"
      : "=r"(d)
      : "r"(pr));
  return d;
}
// Low nibbles of the two 16-bit halves (INT4 codes) -> fp16x2.
__device__ __forceinline__ uint32_t i4_lo_to_h2(uint32_t v) {
  return hsub2((v & 0x000F000Fu) ^ 0x64086408u, 0x64086408u);
}
// Bits 4..7 of the two 16-bit halves (INT4 codes) -> fp16x2.
__device__ __forceinline__ uint32_t i4_hi_to_h2(uint32_t v) {
  return hfma2((v & 0x00F000F0u) ^ 0x64806480u, 0x2C002C00u /* 1/16 */, 0xD480D480u /* -72 */);
}


// 2^e as a float, for -126 <= e <= 127 (exact).
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }

// Unbiased exponent of a positive normal float (floor(log2 x)).
__device__ __forceinline__ int exponent_of(float x) {
  return (int)((__float_as_uint(x) >> 23) & 0xFF) - 127;
}

// FP8: the 8-bit codes are FP8 E4M3 instead of INT8 (same layout, same
// scales; only the code -> fp16 conversion differs).
template <int BITS, bool FP8 = false>
__global__ void __launch_bounds__(kWarps * 32) attn_split_kernel(DevState s, int seq_begin, int batch,
                                                                 const uint16_t* __restrict__ q,
                                                                 float qk_scale_log2, AttnWork w,
                                                                 int spill) {
  using Gm = Geom<BITS>;
  constexpr int STAGES = Gm::kStages;
  constexpr int RB = Gm::kRowBytes;
  __shared__ int cum[kMaxCallBatch + 1];
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
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int r = lane >> 2;
  const int c = lane & 3;
  const long long T = (long long)hkv * cum[batch];
  const int N = gridDim.x;
  const int cta = blockIdx.x;
  long long F = (long long)cta * T / N;
  const long long F1 = (long long)(cta + 1) * T / N;

  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* ring = smem + warp * STAGES * Gm::kStage;

  // per-lane byte offsets of the chunks this lane copies: within a head-page
  // (global) and within a stage (shared); the chunks of one page sit at fixed
  // distances from these, so one asm block copies a page with immediates
  const uint32_t ring_s = smem_u32(smem) + warp * STAGES * Gm::kStage;
  // INT8: bytes 16c and 64 + 16c of rows 2r and 2r+1, so the 4 lanes of a
  // row read whole 32-byte sectors in each copy instruction
  const uint32_t k_goff = BITS == 8 ? (2 * r) * 128 + 16 * c : (2 * r) * 64 + 16 * c;
  const uint32_t v_goff = BITS == 8 ? (4 * c) * 128 + 16 * r : (4 * c) * 64 + 8 * r;
  const uint32_t k_soff = lane * 16;
  const uint32_t v_soff = Gm::kKBytes + (BITS == 8 ? lane * 16 : lane * 8);
  const uint32_t sc_soff = Gm::kKBytes + Gm::kVBytes + 16 * lane;
  const float* sc_gbase = (lane < 4 ? s.k_scale : s.v_scale) + 4 * (lane & 3);

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

    // ---- query fragments (B operand of QK^T), scaled by 2^e_g into fp16 range
    uint32_t bq[8][2];
    float cq0, cq1;
    {
      float qv[32];
      const int g = r;
      if (g < G) {
        // the lane's 32 dims, in the order of its K codes: INT8 dims
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
      if (BITS == 8) {
#pragma unroll
        for (int st = 0; st < 8; ++st) {
          bq[st][0] = pack_half2(qv[4 * st + 0], qv[4 * st + 1]);
          bq[st][1] = pack_half2(qv[4 * st + 2], qv[4 * st + 3]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          bq[2 * i][0] = pack_half2(qv[8 * i + 0], qv[8 * i + 4]);
          bq[2 * i][1] = pack_half2(qv[8 * i + 1], qv[8 * i + 5]);
          bq[2 * i + 1][0] = pack_half2(qv[8 * i + 2], qv[8 * i + 6]);
          bq[2 * i + 1][1] = pack_half2(qv[8 * i + 3], qv[8 * i + 7]);
        }
      }
      const int e0 = __shfl_sync(0xffffffffu, e, (2 * c) * 4);
      const int e1 = __shfl_sync(0xffffffffu, e, (2 * c + 1) * 4);
      cq0 = qk_scale_log2 * pow2i(-e0);
      cq1 = qk_scale_log2 * pow2i(-e1);
    }

    // ---- page pipeline: this warp takes pages pg_a + warp, + kWarps, ...
    const int n_range = pg_e - pg_a;
    const int n_my = n_range > warp ? (n_range - warp + kWarps - 1) / kWarps : 0;
    const int32_t* bt = s.block_table + (size_t)b * s.max_bps;
    uint32_t stage_ok = 0;  // bit k: the page in stage k has a valid block id
    int st_issue = 0;

    auto issue = [&](int k) {
      if (k < n_my) {
        const int page = pg_a + warp + kWarps * k;
        const int blk = bt[page];
        const bool ok = (unsigned)blk < (unsigned)s.num_blocks;
        stage_ok = ok ? (stage_ok | (1u << st_issue)) : (stage_ok & ~(1u << st_issue));
        if (ok) {
          const uint32_t sb = ring_s + st_issue * Gm::kStage;
          const size_t hp = ((size_t)blk * hkv + h) * kPage;
          copy_page<BITS>(sb + k_soff, s.k_codes + hp * RB + k_goff, sb + v_soff, s.v_codes + hp * RB + v_goff);
          if (lane < 8) cp_async16_s(sb + sc_soff, sc_gbase + hp);
        }
      }
      cp_async_commit();
      st_issue = st_issue + 1 == STAGES ? 0 : st_issue + 1;
    };

    float oacc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.0f;
    float m0 = kNegBig, m1 = kNegBig, l0 = 0.0f, l1 = 0.0f;
    int E = 0;
    bool e_set = false;
    float sv_hi = 0.0f;
    float inv2E = 1.0f;
    // logits of this pair, [g][slot]; the lane writes slots (2r, 2r+1) of heads 2c and 2c+1
    float* lg0p = spill && 2 * c < G ? w.logits + ((size_t)pair * G + 2 * c) * w.s_cap + 2 * r : nullptr;
    float* lg1p = spill && 2 * c + 1 < G ? w.logits + ((size_t)pair * G + 2 * c + 1) * w.s_cap + 2 * r : nullptr;

#pragma unroll 1
    for (int k = 0; k < STAGES - 1; ++k) issue(k);

    int st_comp = 0;
#pragma unroll 1
    for (int k = 0; k < n_my; ++k) {
      issue(k + STAGES - 1);
      cp_async_wait<STAGES - 1>();
      __syncwarp();
      const uint8_t* st = ring + st_comp * Gm::kStage;
      const int page = pg_a + warp + kWarps * k;
      const bool blk_ok = (stage_ok >> st_comp) & 1u;
      if (!blk_ok && lane == 0) atomicOr(&s.counters[kCtrStatus], kDevBadBlockId);
      const int slot0 = page * kPage;
      const bool v0 = blk_ok && (slot0 + 2 * r < S);
      const bool v1 = blk_ok && (slot0 + 2 * r + 1 < S);
      const float2 skv = *reinterpret_cast<const float2*>(st + Gm::kKBytes + Gm::kVBytes + 8 * r);
      const float2 svv = *reinterpret_cast<const float2*>(st + Gm::kKBytes + Gm::kVBytes + 64 + 8 * r);

      // ---- S = K_codes . q'  (rows: slots 2r and 2r+1, cols: query heads 2c, 2c+1)
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (BITS == 8) {
        const uint4 ka = *reinterpret_cast<const uint4*>(st + 0 * 512 + lane * 16);
        const uint4 kb2 = *reinterpret_cast<const uint4*>(st + 1 * 512 + lane * 16);
        const uint4 kc = *reinterpret_cast<const uint4*>(st + 2 * 512 + lane * 16);
        const uint4 kd = *reinterpret_cast<const uint4*>(st + 3 * 512 + lane * 16);
        const uint32_t w0[8] = {ka.x, ka.y, ka.z, ka.w, kb2.x, kb2.y, kb2.z, kb2.w};
        const uint32_t w1[8] = {kc.x, kc.y, kc.z, kc.w, kd.x, kd.y, kd.z, kd.w};
#pragma unroll
        for (int stp = 0; stp < 8; ++stp) {
          uint32_t a0, a1, a2, a3;
          if (FP8) {
            e4m3x4_to_h2(w0[stp], a0, a2);
            e4m3x4_to_h2(w1[stp], a1, a3);
          } else {
            i8x4_to_h2(w0[stp] ^ 0x80808080u, a0, a2);
            i8x4_to_h2(w1[stp] ^ 0x80808080u, a1, a3);
          }
          mma16816(acc, a0, a1, a2, a3, bq[stp][0], bq[stp][1]);
        }
      } else {
        const uint4 ka = *reinterpret_cast<const uint4*>(st + 0 * 512 + lane * 16);
        const uint4 kb2 = *reinterpret_cast<const uint4*>(st + 1 * 512 + lane * 16);
        const uint32_t w0[4] = {ka.x, ka.y, ka.z, ka.w};
        const uint32_t w1[4] = {kb2.x, kb2.y, kb2.z, kb2.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t x0 = w0[i], x1 = w1[i];
          const uint32_t x0s = x0 >> 8, x1s = x1 >> 8;
          mma16816(acc, i4_lo_to_h2(x0), i4_lo_to_h2(x1), i4_hi_to_h2(x0), i4_hi_to_h2(x1), bq[2 * i][0],
                   bq[2 * i][1]);
          mma16816(acc, i4_lo_to_h2(x0s), i4_lo_to_h2(x1s), i4_hi_to_h2(x0s), i4_hi_to_h2(x1s),
                   bq[2 * i + 1][0], bq[2 * i + 1][1]);
        }
      }
      const float lg0 = v0 ? acc[0] * skv.x * cq0 : -INFINITY;  // slot 2r,   head 2c
      const float lg1 = v0 ? acc[1] * skv.x * cq1 : -INFINITY;  // slot 2r,   head 2c+1
      const float lg2 = v1 ? acc[2] * skv.y * cq0 : -INFINITY;  // slot 2r+1, head 2c
      const float lg3 = v1 ? acc[3] * skv.y * cq1 : -INFINITY;  // slot 2r+1, head 2c+1
      if (lg0p) *reinterpret_cast<float2*>(lg0p + slot0) = make_float2(lg0, lg2);
      if (lg1p) *reinterpret_cast<float2*>(lg1p + slot0) = make_float2(lg1, lg3);

      // ---- lazy online softmax: reduce and rescale only when some lane's
      // logit exceeds the running max by kLazy, or a V scale outgrows 2^(E+4)
      const float svl = fmaxf(v0 ? svv.x : 0.0f, v1 ? svv.y : 0.0f);
      const bool need = fmaxf(lg0, lg2) > m0 + kLazy || fmaxf(lg1, lg3) > m1 + kLazy || svl > sv_hi ||
                        (!e_set && svl > 0.0f);
      if (__any_sync(0xffffffffu, need)) {
        float tm0 = fmaxf(lg0, lg2), tm1 = fmaxf(lg1, lg3), svm = svl;
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
      const float sn0 = v0 ? svv.x * inv2E : 0.0f;
      const float sn1 = v1 ? svv.y * inv2E : 0.0f;
      const float p0 = fast_exp2(lg0 - m0), p1 = fast_exp2(lg1 - m1);
      const float p2 = fast_exp2(lg2 - m0), p3 = fast_exp2(lg3 - m1);
      l0 += p0 + p2;
      l1 += p1 + p3;
      const uint32_t pb0 = movmatrix_t(pack_half2(p0 * sn0, p1 * sn0));
      const uint32_t pb1 = movmatrix_t(pack_half2(p2 * sn1, p3 * sn1));

      // ---- O^T += V_codes^T . P~^T   (rows: head-dim 16r + 2j (+1), cols: query heads)
      if (BITS == 8) {
        const uint4 r0 = *reinterpret_cast<const uint4*>(st + Gm::kKBytes + 0 * 512 + lane * 16);
        const uint4 r1 = *reinterpret_cast<const uint4*>(st + Gm::kKBytes + 1 * 512 + lane * 16);
        const uint4 r2 = *reinterpret_cast<const uint4*>(st + Gm::kKBytes + 2 * 512 + lane * 16);
        const uint4 r3 = *reinterpret_cast<const uint4*>(st + Gm::kKBytes + 3 * 512 + lane * 16);
        const uint32_t x0[4] = {r0.x, r0.y, r0.z, r0.w};  // slot 4c
        const uint32_t x1[4] = {r1.x, r1.y, r1.z, r1.w};  // slot 4c+1
        const uint32_t x2[4] = {r2.x, r2.y, r2.z, r2.w};  // slot 4c+2
        const uint32_t x3[4] = {r3.x, r3.y, r3.z, r3.w};  // slot 4c+3
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int j = 2 * wd + half;
            uint32_t a0, a1, a2, a3;
            if (FP8) {
              a0 = e4m3_pair_to_h2(x0[wd], x2[wd], 2 * half);
              a1 = e4m3_pair_to_h2(x0[wd], x2[wd], 2 * half + 1);
              a2 = e4m3_pair_to_h2(x1[wd], x3[wd], 2 * half);
              a3 = e4m3_pair_to_h2(x1[wd], x3[wd], 2 * half + 1);
            } else {
              const uint32_t sa = (2 * half) | ((2 * half) << 4) | ((4 + 2 * half) << 8) | ((4 + 2 * half) << 12);
              const uint32_t sb =
                  (2 * half + 1) | ((2 * half + 1) << 4) | ((5 + 2 * half) << 8) | ((5 + 2 * half) << 12);
              a0 = i8_pair_to_h2(x0[wd], x2[wd], sa);
              a1 = i8_pair_to_h2(x0[wd], x2[wd], sb);
              a2 = i8_pair_to_h2(x1[wd], x3[wd], sa);
              a3 = i8_pair_to_h2(x1[wd], x3[wd], sb);
            }
            mma16816(oacc[j], a0, a1, a2, a3, pb0, pb1);
          }
        }
      } else {
        const uint2 r0 = *reinterpret_cast<const uint2*>(st + Gm::kKBytes + 0 * 256 + lane * 8);
        const uint2 r1 = *reinterpret_cast<const uint2*>(st + Gm::kKBytes + 1 * 256 + lane * 8);
        const uint2 r2 = *reinterpret_cast<const uint2*>(st + Gm::kKBytes + 2 * 256 + lane * 8);
        const uint2 r3 = *reinterpret_cast<const uint2*>(st + Gm::kKBytes + 3 * 256 + lane * 8);
        const uint32_t x0[2] = {r0.x, r0.y};
        const uint32_t x1[2] = {r1.x, r1.y};
        const uint32_t x2[2] = {r2.x, r2.y};
        const uint32_t x3[2] = {r3.x, r3.y};
#pragma unroll
        for (int u = 0; u < 2; ++u) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int j = 4 * u + kk;
            const uint32_t sel = kk | (kk << 4) | ((4 + kk) << 8) | ((4 + kk) << 12);
            const uint32_t v02 = prmt(x0[u], x2[u], sel);
            const uint32_t v13 = prmt(x1[u], x3[u], sel);
            mma16816(oacc[j], i4_lo_to_h2(v02), i4_hi_to_h2(v02), i4_lo_to_h2(v13), i4_hi_to_h2(v13), pb0,
                     pb1);
          }
        }
      }
      st_comp = st_comp + 1 == STAGES ? 0 : st_comp + 1;
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
      float* o0 = sm_o + ((size_t)warp * kMaxGroup + 2 * c) * kHeadDim + 16 * r;
      float* o1 = o0 + kHeadDim;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        o0[2 * j] = oacc[j][0] * f2E;
        o0[2 * j + 1] = oacc[j][2] * f2E;
        o1[2 * j] = oacc[j][1] * f2E;
        o1[2 * j + 1] = oacc[j][3] * f2E;
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
// write the bf16 outputs of its G query heads; with H2O on, add this step's
// probabilities to the sink scores and to every pool slot's score.
__global__ void __launch_bounds__(kMergeThreads, 2) attn_merge_kernel(DevState s, int seq_begin, int batch,
                                                                     const uint16_t* __restrict__ q,
                                                                     uint16_t* __restrict__ out,
                                                                     float qk_scale_log2, AttnWork w, int accumulate) {
  __shared__ int cum[kMaxCallBatch + 1];
  __shared__ MergeShared ms;
  __shared__ int32_t sh_bt[kMergeBtStage];
  pages_prefix(s, seq_begin, batch, cum);
  const int h = blockIdx.x;
  const int bl = blockIdx.y;
  merge_phase(s, seq_begin, batch, cum, h, bl, q, out, qk_scale_log2, w, accumulate != 0, ms);
  if (!accumulate) return;
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
                                   float qk_scale_log2, const AttnWork& w, bool accumulate, cudaStream_t st) {
  dim3 grid(s.hkv, batch);
  attn_merge_kernel<<<grid, kMergeThreads, 0, st>>>(s, seq_begin, batch, q, out, qk_scale_log2, w, accumulate ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace kvc
