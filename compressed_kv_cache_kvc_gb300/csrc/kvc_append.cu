// Quantise-on-write of new tokens into the paged pool.
//
// Per (token, KV head) row of K and of V ("KV Cache optimization techniques",
// section 1.2 per-token quantisation; Technical Report section 3.2): amax over
// the 128 values, scale = amax / qmax in IEEE fp32, code = round-half-even of
// x / scale (IEEE fp32 division), clamped.  Positions 0..3 are attention sinks
// and are copied unchanged in bf16 (Technical Report section 3.2).
//
// One CTA per sequence: thread 0 takes the pages the new tokens need from the
// device free-block stack and advances the sequence lengths; after a barrier
// every warp quantises rows (one warp per 128-value row, 4 values per lane).
//
// Hybrid precision ("KV Cache optimization techniques" section 1.3): with a
// window of W positions, a new token goes to the bf16 ring of its (sequence,
// KV head), slot (position - 4) mod W, and enters the pool, quantised from
// the ring, only when a later append pushes it out of the window.
#include "kvc_internal.h"
#include "kvc_mma.h"

namespace kvc {
namespace {

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// Quantise one 128-value row (4 values per lane, one warp) into pool slot
// `slot` of a sequence's KV head h, `blk` the block id of the slot's page
// (from its block-table row): codes, scale, and for K the position and the
// initial score.  Integer codes, or with E4M3 codes (s.fp8) scale =
// amax / 448 and each x / scale converted to FP8.
// Four fp32 values -> four FP8 E4M3 codes (byte i = value i), rounded to
// nearest even and saturated to +-448 by the conversion instruction (which
// packs its first source into the upper byte).
__device__ __forceinline__ uint32_t e4m3x4(float y0, float y1, float y2, float y3) {
  uint32_t w;
  asm("{\n .reg .b16 l, h;\n"
      " cvt.rn.satfinite.e4m3x2.f32 l, %2, %1;\n"
      " cvt.rn.satfinite.e4m3x2.f32 h, %4, %3;\n"
      " mov.b32 %0, {l, h};\n}"
      : "=r"(w)
      : "f"(y0), "f"(y1), "f"(y2), "f"(y3));
  return w;
}

template <int BITS>
__device__ __forceinline__ void quantize_row_blk(const DevState& s, int blk, int h, int kv, int slot, int p,
                                                 float score, uint2 raw, int lane) {
  constexpr float kQmax = BITS == 8 ? 127.0f : 7.0f;
  constexpr int kLo = BITS == 8 ? -127 : -8;
  constexpr int kHi = BITS == 8 ? 127 : 7;
  float x[4];
  x[0] = bf16_to_f32(raw.x & 0xFFFFu);
  x[1] = bf16_to_f32(raw.x >> 16);
  x[2] = bf16_to_f32(raw.y & 0xFFFFu);
  x[3] = bf16_to_f32(raw.y >> 16);
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const bool fp8 = BITS == 8 && s.fp8;
  const float scale = __fdiv_rn(amax, fp8 ? 448.0f : kQmax);
  int c[4] = {0, 0, 0, 0};
  if (!fp8) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int q = 0;
      if (scale > 0.0f) q = __float2int_rn(__fdiv_rn(x[e], scale));
      c[e] = min(max(q, kLo), kHi);
    }
  }
  const int off = slot % kPage;
  if ((unsigned)blk >= (unsigned)s.num_blocks) {
    if (lane == 0) atomicOr(&s.counters[kCtrStatus], kDevBadBlockId);
    return;
  }
  const size_t sidx = ((size_t)blk * s.hkv + h) * kPage + off;
  uint8_t* codes = (kv ? s.v_codes : s.k_codes) + sidx * s.row_bytes;
  if (fp8) {
    float y[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] = scale > 0.0f ? __fdiv_rn(x[e], scale) : 0.0f;
    *reinterpret_cast<uint32_t*>(codes + lane * 4) = e4m3x4(y[0], y[1], y[2], y[3]);
  } else if (BITS == 8) {
    const uint32_t packed = (uint32_t)(c[0] & 0xFF) | ((uint32_t)(c[1] & 0xFF) << 8) |
                            ((uint32_t)(c[2] & 0xFF) << 16) | ((uint32_t)(c[3] & 0xFF) << 24);
    *reinterpret_cast<uint32_t*>(codes + lane * 4) = packed;
  } else {
    const uint32_t packed = (uint32_t)(c[0] & 0xF) | ((uint32_t)(c[1] & 0xF) << 4) |
                            ((uint32_t)(c[2] & 0xF) << 8) | ((uint32_t)(c[3] & 0xF) << 12);
    *reinterpret_cast<uint16_t*>(codes + lane * 2) = (uint16_t)packed;
  }
  if (lane == 0) {
    (kv ? s.v_scale : s.k_scale)[sidx] = scale;
    if (kv == 0) {
      s.slot_pos[sidx] = p;
      s.score[sidx] = score;
    }
  }
}

template <int BITS>
__global__ void __launch_bounds__(512) append_kernel(DevState s, int seq_begin, int n_new,
                                                     const uint16_t* __restrict__ kin,
                                                     const uint16_t* __restrict__ vin) {
  const int bl = blockIdx.x;
  const int b = seq_begin + bl;
  constexpr int kPagesStaged = 8;
  __shared__ int sh_slots, sh_pos, sh_ok, sh_lo, sh_hi;
  __shared__ int sh_blk[kPagesStaged];  // block ids of the pages this append writes, from page slots / 16
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int hkv = s.hkv;
  const int W = s.ring;
  // this warp's first new-token row (row = warp), loaded while thread 0 takes
  // the pages: the input does not depend on them
  const int rows_new = n_new * hkv * 2;
  uint2 raw0 = make_uint2(0u, 0u);
  if (warp < rows_new) {
    const int h = (warp >> 1) % hkv;
    const int i = (warp >> 1) / hkv;
    const uint16_t* src = ((warp & 1) ? vin : kin) + (((size_t)bl * hkv + h) * n_new + i) * kHeadDim;
    raw0 = *reinterpret_cast<const uint2*>(src + lane * 4);
  }
  if (threadIdx.x == 0) {
    const int slots = s.seq_slots[b];
    const int pos = s.seq_pos[b];
    int lo, hi;  // positions that enter the pool
    pool_range(pos, n_new, s.ring, &lo, &hi);
    const int new_slots = slots + (hi - lo);
    const int old_pages = (slots + kPage - 1) / kPage;
    const int new_pages = (new_slots + kPage - 1) / kPage;
    const int need = new_pages - old_pages;
    int ok = 1;
    int32_t* row = s.block_table + (size_t)b * s.max_bps;
    if (new_pages > s.max_bps) {
      atomicOr(&s.counters[kCtrStatus], kDevTableOverflow);
      ok = 0;
    } else if (need > 0) {
      const int top = atomicSub(&s.counters[kCtrFreeTop], need);
      if (top - need < 0 || top > s.num_blocks) {
        atomicAdd(&s.counters[kCtrFreeTop], need);
        atomicOr(&s.counters[kCtrStatus], kDevOutOfBlocks);
        ok = 0;
      } else {
        for (int j = 0; j < need; ++j) {
          const int blk = s.free_stack[top - 1 - j];
          row[old_pages + j] = blk;
          const int k = old_pages + j - slots / kPage;
          if (k < kPagesStaged) sh_blk[k] = blk;
        }
      }
    }
    // the partly filled page the first new slot lands in, if any
    if (ok && slots % kPage != 0 && new_slots > slots) sh_blk[0] = row[slots / kPage];
    if (ok) {
      s.seq_slots[b] = new_slots;
      s.seq_pos[b] = pos + n_new;
    }
    sh_slots = slots;
    sh_pos = pos;
    sh_ok = ok;
    sh_lo = lo;
    sh_hi = hi;
  }
  __syncthreads();
  if (!sh_ok) return;
  // block id of pool slot `slot` of this append (slots [sh_slots, new slots))
  auto blk_of = [&](int slot) {
    const int k = slot / kPage - sh_slots / kPage;
    return k < kPagesStaged ? sh_blk[k] : s.block_table[(size_t)b * s.max_bps + slot / kPage];
  };

  // ---- hybrid precision: the window tokens this append pushes out (positions
  // [lo, min(pos, hi)), all in the ring) are quantised into the pool with the
  // score they gathered there, before any new token overwrites their slots
  if (W > 0) {
    const int n_aged = max(0, min(sh_pos, sh_hi) - sh_lo);
    for (int row = warp; row < n_aged * hkv * 2; row += nwarps) {
      const int kv = row & 1;
      const int h = (row >> 1) % hkv;
      const int a = sh_lo + (row >> 1) / hkv;
      const size_t ridx = ((size_t)b * hkv + h) * W + (a - kSinks) % W;
      const uint16_t* src = (kv ? s.ring_v : s.ring_k) + ridx * kHeadDim;
      const uint2 raw = *reinterpret_cast<const uint2*>(src + lane * 4);
      const int slot = sh_slots + (a - sh_lo);
      quantize_row_blk<BITS>(s, blk_of(slot), h, kv, slot, a, s.ring_score[ridx], raw, lane);
    }
    __syncthreads();
  }

  // ---- the new tokens: sinks, pool (quantised), or the window ring (bf16)
  for (int row = warp; row < rows_new; row += nwarps) {
    const int kv = row & 1;
    const int h = (row >> 1) % hkv;
    const int i = (row >> 1) / hkv;
    const uint16_t* src = (kv ? vin : kin) + (((size_t)bl * hkv + h) * n_new + i) * kHeadDim;
    const uint2 raw = row == warp ? raw0 : *reinterpret_cast<const uint2*>(src + lane * 4);
    const int p = sh_pos + i;
    if (p < kSinks) {
      uint16_t* dst = (kv ? s.sink_v : s.sink_k) + (((size_t)b * hkv + h) * kSinks + p) * kHeadDim;
      *reinterpret_cast<uint2*>(dst + lane * 4) = raw;
      if (kv == 0 && lane == 0) s.sink_score[((size_t)b * hkv + h) * kSinks + p] = 0.0f;
    } else if (p < sh_hi) {
      const int slot = sh_slots + (p - sh_lo);
      quantize_row_blk<BITS>(s, blk_of(slot), h, kv, slot, p, 0.0f, raw, lane);
    } else {
      const size_t ridx = ((size_t)b * hkv + h) * W + (p - kSinks) % W;
      uint16_t* dst = (kv ? s.ring_v : s.ring_k) + ridx * kHeadDim;
      *reinterpret_cast<uint2*>(dst + lane * 4) = raw;
      if (kv == 0 && lane == 0) s.ring_score[ridx] = 0.0f;
    }
  }
}

// Bulk appends (a prompt) run as two launches: append_alloc_kernel, one
// warp per sequence, takes the pages and advances the lengths exactly as
// append_kernel's first thread does and leaves the old lengths in the plan
// scratch (slots -1 when it failed); append_rows_kernel then spreads the
// rows over (token chunk, sequence) CTAs.  Only for appends that push no
// window token into the pool, so no row reads what another CTA writes.
constexpr int kBulkTokens = 32;  // most tokens per CTA of append_rows_kernel (at most 3 pool pages)
constexpr int kBulkWarps = 16;
constexpr int kBulkStages = 6;  // units a warp keeps in flight (1 KB each)
constexpr int kBulkSmem = kBulkWarps * kBulkStages * 1024;

// One warp per sequence: lane 0 takes the pages off the free stack, the
// lanes copy their block ids into the sequence's block-table row.
__global__ void append_alloc_kernel(DevState s, int seq_begin, int batch, int n_new) {
  const int lane = threadIdx.x & 31;
  const int bl = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (bl >= batch) return;  // the same for the whole warp
  const int b = seq_begin + bl;
  const int slots = s.seq_slots[b];
  const int pos = s.seq_pos[b];
  int lo, hi;
  pool_range(pos, n_new, s.ring, &lo, &hi);
  const int new_slots = slots + (hi - lo);
  const int old_pages = (slots + kPage - 1) / kPage;
  const int new_pages = (new_slots + kPage - 1) / kPage;
  const int need = new_pages - old_pages;
  int ok = 1;
  if (new_pages > s.max_bps) {
    if (lane == 0) atomicOr(&s.counters[kCtrStatus], kDevTableOverflow);
    ok = 0;
  } else if (need > 0) {
    int top = 0;
    if (lane == 0) {
      top = atomicSub(&s.counters[kCtrFreeTop], need);
      if (top - need < 0 || top > s.num_blocks) {
        atomicAdd(&s.counters[kCtrFreeTop], need);
        atomicOr(&s.counters[kCtrStatus], kDevOutOfBlocks);
        top = -1;
      }
    }
    top = __shfl_sync(0xffffffffu, top, 0);
    if (top < 0) {
      ok = 0;
    } else {
      int32_t* row = s.block_table + (size_t)b * s.max_bps;
      for (int j = lane; j < need; j += 32) row[old_pages + j] = s.free_stack[top - 1 - j];
    }
  }
  if (lane == 0) {
    if (ok) {
      s.seq_slots[b] = new_slots;
      s.seq_pos[b] = pos + n_new;
    }
    s.plan[2 * b] = ok ? slots : -1;
    s.plan[2 * b + 1] = pos;
  }
}

// Integer codes of 8 values of a row, as words whose low byte is the
// two's-complement 8-bit code and whose low nibble is the 4-bit one
// (0x4B400000 + code: the fp32 bit pattern of 1.5 * 2^23 + code).
//
// code = round-half-even(x / scale) with x / scale the IEEE fp32 quotient,
// clamped, as in quantize_row.  Here the code comes, where that decides it,
// from the exact product P = x * inv, inv an approximate reciprocal of the
// scale (relative error at most 2^-23, one ulp): P differs from the rounded
// quotient by at most 2^-23 |x / scale| + 2^-24 |x / scale| < 2^-14.4,
// because |x| <= amax gives |x / scale| <= qmax (1 + 2^-23) < 128 (the scale
// is a normal number here; a subnormal one has an infinite reciprocal under
// ftz).  One fused multiply-add rounds P + 1.5 * 2^23 to the integer r
// nearest P (round to nearest even in the binade of unit spacing); a second
// gives P - r.  Where |P - r| < 1/2 - 2^-12 the quotient lies in the same
// unit interval around r and rounds to r, and |r| <= qmax needs no clamp.
// Elsewhere (P within about 2^-12 of a half-integer, or not finite) the
// division decides.  About one value in 2^11 takes that path.
__device__ __forceinline__ float rcp_approx_ftz(float a) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
  return r;
}

template <int BITS>
__device__ __forceinline__ void int_codes8(const float* x, float scale, float inv, uint32_t (&w)[8]) {
  constexpr float kM = 12582912.0f;  // 1.5 * 2^23
  constexpr float kNear = 0.5f - 0x1p-12f;
  constexpr int kLo = BITS == 8 ? -127 : -8;
  constexpr int kHi = BITS == 8 ? 127 : 7;
  bool slow = false;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float sm = __fmaf_rn(x[e], inv, kM);
    w[e] = __float_as_uint(sm);
    slow |= !(fabsf(__fmaf_rn(x[e], inv, -__fadd_rn(sm, -kM))) < kNear);
  }
  if (slow) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float r = __fadd_rn(__fmaf_rn(x[e], inv, kM), -kM);
      if (!(fabsf(__fmaf_rn(x[e], inv, -r)) < kNear)) {
        const int q = scale > 0.0f ? min(max(__float2int_rn(__fdiv_rn(x[e], scale)), kLo), kHi) : 0;
        w[e] = 0x4B400000u + (uint32_t)q;
      }
    }
  }
}

// the low bytes of four words, in order
__device__ __forceinline__ uint32_t low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// Rows spread over (token chunk, sequence) CTAs.  A unit is 4 adjacent
// tokens of one (KV head, K or V): 4 rows of 128 values, one per quarter of
// a warp; a lane takes dims 8j .. 8j + 7 and 64 + 8j .. 64 + 8j + 7 of its
// row, so a unit is one 1 KB run of the input.  Each warp streams its units
// (u = warp, warp + 16, ...) through a ring of kBulkStages 1 KB stages in
// shared memory with cp.async: every lane copies its own 32 bytes of a unit
// and later reads back exactly those, so the ring needs no barrier, only
// the lane's own wait for its copy group.  Stage layout: the lanes' first
// 16-byte chunks, then their second ones (conflict-free reads).  The unit
// indices advance by the warp count without divisions.
template <int BITS>
__global__ void __launch_bounds__(kBulkWarps * 32, 2) append_rows_kernel(DevState s, int seq_begin, int n_new,
                                                                          int chunk,
                                                                          const uint16_t* __restrict__ kin,
                                                                          const uint16_t* __restrict__ vin) {
  using namespace codes;
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ int sh_blk[4];
  const int bl = blockIdx.y;
  const int b = seq_begin + bl;
  const int slots = s.plan[2 * b];
  if (slots < 0) return;  // the same for the whole CTA
  const int pos = s.plan[2 * b + 1];
  int lo, hi;
  pool_range(pos, n_new, s.ring, &lo, &hi);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int qr = lane >> 3;  // which token of the unit
  const int ql = lane & 7;   // which dims of its row
  const int hkv = s.hkv;
  const int W = s.ring;
  const int t0 = blockIdx.x * chunk;
  const int nt = min(chunk, n_new - t0);
  const int nquad = (nt + 3) >> 2;
  const int units = nquad * hkv * 2;  // unit u: token quad u % nquad, (KV head, K or V) u / nquad
  const int dq = kBulkWarps / nquad, dr = kBulkWarps % nquad;
  const bool fp8 = BITS == 8 && s.fp8;

  // the block ids of the (at most 3) pool pages this chunk's tokens land in
  const int pf = max(pos + t0, lo), pl = min(pos + t0 + nt, hi);  // pool positions [pf, pl)
  const int page0 = pf < pl ? (slots + (pf - lo)) / kPage : 0;
  if (threadIdx.x < 4) {
    const int pg = page0 + threadIdx.x;
    sh_blk[threadIdx.x] = pf < pl && pg <= (slots + (pl - 1 - lo)) / kPage ? s.block_table[(size_t)b * s.max_bps + pg] : -1;
  }
  __syncthreads();

  const uint32_t ring_s = smem_u32(ring) + warp * (kBulkStages * 1024) + 16 * lane;
  // issue cursor: unit warp + ki * 16 is (iquad, ihk), into stage istage
  int iquad = warp % nquad, ihk = warp / nquad, istage = 0;
  auto issue = [&](int ki) {
    const int tok = t0 + 4 * iquad + qr;
    const bool ok = warp + ki * kBulkWarps < units && tok < t0 + nt;
    const uint16_t* src =
        ((ihk & 1) ? vin : kin) + (((size_t)bl * hkv + (ihk >> 1)) * n_new + (ok ? tok : 0)) * kHeadDim + 8 * ql;
    const uint32_t dst = ring_s + istage * 1024;
    cp_async16_if(ok, dst, src);
    cp_async16_if(ok, dst + 512, src + 64);
    cp_async_commit();
    istage = istage == kBulkStages - 1 ? 0 : istage + 1;
    iquad += dr;
    ihk += dq;
    if (iquad >= nquad) {
      iquad -= nquad;
      ++ihk;
    }
  };
#pragma unroll 1
  for (int ki = 0; ki < kBulkStages - 1; ++ki) issue(ki);

  int quad = warp % nquad, hk = warp / nquad, stage = 0;  // processing cursor
#pragma unroll 1
  for (int k = 0; warp + k * kBulkWarps < units; ++k) {
    cp_async_wait<kBulkStages - 2>();  // this lane's copies of unit k have landed
    issue(k + kBulkStages - 1);        // into the stage unit k - 1 was read from
    const uint32_t st = ring_s + stage * 1024;
    uint4 r0, r1;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r0.x), "=r"(r0.y), "=r"(r0.z), "=r"(r0.w) : "r"(st));
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r1.x), "=r"(r1.y), "=r"(r1.z), "=r"(r1.w)
                 : "r"(st + 512));
    const int tok = t0 + 4 * quad + qr;
    const int kv = hk & 1;
    const int h = hk >> 1;
    stage = stage == kBulkStages - 1 ? 0 : stage + 1;
    quad += dr;
    hk += dq;
    if (quad >= nquad) {
      quad -= nquad;
      ++hk;
    }

    const uint32_t wd[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
    float x[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[2 * i] = __uint_as_float(wd[i] << 16);
      x[2 * i + 1] = __uint_as_float(wd[i] & 0xFFFF0000u);
    }
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (tok >= t0 + nt) continue;  // past the chunk's last token (its lanes read nothing)
    const int p = pos + tok;
    if (p < kSinks) {
      const size_t si = ((size_t)b * hkv + h) * kSinks + p;
      uint16_t* dst = (kv ? s.sink_v : s.sink_k) + si * kHeadDim + 8 * ql;
      *reinterpret_cast<uint4*>(dst) = r0;
      *reinterpret_cast<uint4*>(dst + 64) = r1;
      if (kv == 0 && ql == 0) s.sink_score[si] = 0.0f;
      continue;
    }
    if (p >= hi) {
      const size_t ridx = ((size_t)b * hkv + h) * W + (p - kSinks) % W;
      uint16_t* dst = (kv ? s.ring_v : s.ring_k) + ridx * kHeadDim + 8 * ql;
      *reinterpret_cast<uint4*>(dst) = r0;
      *reinterpret_cast<uint4*>(dst + 64) = r1;
      if (kv == 0 && ql == 0) s.ring_score[ridx] = 0.0f;
      continue;
    }
    const int slot = slots + (p - lo);
    const int blk = sh_blk[slot / kPage - page0];
    if ((unsigned)blk >= (unsigned)s.num_blocks) {
      if (ql == 0) atomicOr(&s.counters[kCtrStatus], kDevBadBlockId);
      continue;
    }
    const float scale = __fdiv_rn(amax, fp8 ? 448.0f : (BITS == 8 ? 127.0f : 7.0f));
    // scale 0 (an all-zero row) gives an infinite reciprocal: every value
    // then takes the slow path, which gives code 0
    const float inv = rcp_approx_ftz(scale);
    const size_t sidx = ((size_t)blk * hkv + h) * kPage + slot % kPage;
    uint8_t* codes = (kv ? s.v_codes : s.k_codes) + sidx * s.row_bytes;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {  // dims 8 ql.. (hh 0) and 64 + 8 ql.. (hh 1)
      const float* xh = x + 8 * hh;
      if (fp8) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = scale > 0.0f ? __fdiv_rn(xh[e], scale) : 0.0f;
        *reinterpret_cast<uint2*>(codes + 64 * hh + 8 * ql) =
            make_uint2(e4m3x4(y[0], y[1], y[2], y[3]), e4m3x4(y[4], y[5], y[6], y[7]));
      } else {
        uint32_t wc[8];
        int_codes8<BITS>(xh, scale, inv, wc);
        if (BITS == 8) {
          *reinterpret_cast<uint2*>(codes + 64 * hh + 8 * ql) =
              make_uint2(low_bytes(wc[0], wc[1], wc[2], wc[3]), low_bytes(wc[4], wc[5], wc[6], wc[7]));
        } else {
          // byte i: the nibble of value 2i low, of value 2i + 1 high
          const uint32_t ev = low_bytes(wc[0], wc[2], wc[4], wc[6]);
          const uint32_t od = low_bytes(wc[1], wc[3], wc[5], wc[7]);
          *reinterpret_cast<uint32_t*>(codes + 32 * hh + 4 * ql) = (ev & 0x0F0F0F0Fu) | ((od & 0x0F0F0F0Fu) << 4);
        }
      }
    }
    if (ql == 0) {
      (kv ? s.v_scale : s.k_scale)[sidx] = scale;
      if (kv == 0) {
        s.slot_pos[sidx] = p;
        s.score[sidx] = 0.0f;
      }
    }
  }
  cp_async_wait<0>();  // (only empty groups can be pending here)
}

__global__ void fill_free_stack_kernel(int32_t* stack, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) stack[i] = n - 1 - i;
}

}  // namespace

cudaError_t launch_append_bulk(const DevState& s, int seq_begin, int batch, int n_new, const uint16_t* k,
                               const uint16_t* v, cudaStream_t st) {
  append_alloc_kernel<<<(batch * 32 + 127) / 128, 128, 0, st>>>(s, seq_begin, batch, n_new);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  static int done8[64] = {0}, done4[64] = {0};
  e = s.bits == 8 ? opt_in_smem(reinterpret_cast<const void*>(append_rows_kernel<8>), kBulkSmem, done8)
                  : opt_in_smem(reinterpret_cast<const void*>(append_rows_kernel<4>), kBulkSmem, done4);
  if (e != cudaSuccess) return e;
  // tokens per CTA: kBulkTokens, halved (down to one 4-token unit) while
  // the grid would not give every SM two CTAs (short prompts)
  static int sms[64] = {0};
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || sms[dev] == 0) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev < 64) sms[dev] = n;
  }
  const long long want = 2LL * (dev < 64 ? sms[dev] : 152);
  int chunk = kBulkTokens;
  while (chunk > 4 && (long long)((n_new + chunk - 1) / chunk) * batch < want) chunk /= 2;
  const dim3 grid((n_new + chunk - 1) / chunk, batch);
  if (s.bits == 8)
    append_rows_kernel<8><<<grid, kBulkWarps * 32, kBulkSmem, st>>>(s, seq_begin, n_new, chunk, k, v);
  else
    append_rows_kernel<4><<<grid, kBulkWarps * 32, kBulkSmem, st>>>(s, seq_begin, n_new, chunk, k, v);
  return cudaGetLastError();
}

cudaError_t launch_append(const DevState& s, int seq_begin, int batch, int n_new, const uint16_t* k,
                          const uint16_t* v, cudaStream_t st) {
  const int rows = n_new * s.hkv * 2;
  int threads = 32 * min(16, max(1, rows));
  if (s.bits == 8)
    append_kernel<8><<<batch, threads, 0, st>>>(s, seq_begin, n_new, k, v);
  else
    append_kernel<4><<<batch, threads, 0, st>>>(s, seq_begin, n_new, k, v);
  return cudaGetLastError();
}

cudaError_t launch_fill_free_stack(const DevState& s, cudaStream_t st) {
  fill_free_stack_kernel<<<64, 256, 0, st>>>(s.free_stack, s.num_blocks);
  return cudaGetLastError();
}

}  // namespace kvc
