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

namespace kvc {
namespace {

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// Quantise one 128-value row (4 values per lane, one warp) into pool slot
// `slot` of (sequence b, KV head h): codes, scale, and for K the position and
// the initial score.  Integer codes, or with E4M3 codes (s.fp8) scale =
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
__device__ __forceinline__ void quantize_row(const DevState& s, int b, int h, int kv, int slot, int p, float score,
                                             uint2 raw, int lane) {
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
  const int page = slot / kPage;
  const int off = slot % kPage;
  const int blk = s.block_table[(size_t)b * s.max_bps + page];
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
  __shared__ int sh_slots, sh_pos, sh_ok, sh_lo, sh_hi;
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
        int32_t* row = s.block_table + (size_t)b * s.max_bps;
        for (int j = 0; j < need; ++j) row[old_pages + j] = s.free_stack[top - 1 - j];
      }
    }
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

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int hkv = s.hkv;
  const int W = s.ring;

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
      quantize_row<BITS>(s, b, h, kv, sh_slots + (a - sh_lo), a, s.ring_score[ridx], raw, lane);
    }
    __syncthreads();
  }

  // ---- the new tokens: sinks, pool (quantised), or the window ring (bf16)
  for (int row = warp; row < n_new * hkv * 2; row += nwarps) {
    const int kv = row & 1;
    const int h = (row >> 1) % hkv;
    const int i = (row >> 1) / hkv;
    const uint16_t* src = (kv ? vin : kin) + (((size_t)bl * hkv + h) * n_new + i) * kHeadDim;
    const uint2 raw = *reinterpret_cast<const uint2*>(src + lane * 4);
    const int p = sh_pos + i;
    if (p < kSinks) {
      uint16_t* dst = (kv ? s.sink_v : s.sink_k) + (((size_t)b * hkv + h) * kSinks + p) * kHeadDim;
      *reinterpret_cast<uint2*>(dst + lane * 4) = raw;
      if (kv == 0 && lane == 0) s.sink_score[((size_t)b * hkv + h) * kSinks + p] = 0.0f;
    } else if (p < sh_hi) {
      quantize_row<BITS>(s, b, h, kv, sh_slots + (p - sh_lo), p, 0.0f, raw, lane);
    } else {
      const size_t ridx = ((size_t)b * hkv + h) * W + (p - kSinks) % W;
      uint16_t* dst = (kv ? s.ring_v : s.ring_k) + ridx * kHeadDim;
      *reinterpret_cast<uint2*>(dst + lane * 4) = raw;
      if (kv == 0 && lane == 0) s.ring_score[ridx] = 0.0f;
    }
  }
}

// Bulk appends (a prompt) run as two launches: append_alloc_kernel, one
// thread per sequence, takes the pages and advances the lengths exactly as
// append_kernel's first thread does and leaves the old lengths in the plan
// scratch (slots -1 when it failed); append_rows_kernel then spreads the
// rows over (token chunk, sequence) CTAs.  Only for appends that push no
// window token into the pool, so no row reads what another CTA writes.
constexpr int kBulkTokens = 64;  // tokens per CTA of append_rows_kernel

__global__ void append_alloc_kernel(DevState s, int seq_begin, int batch, int n_new) {
  const int bl = blockIdx.x * blockDim.x + threadIdx.x;
  if (bl >= batch) return;
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
    atomicOr(&s.counters[kCtrStatus], kDevTableOverflow);
    ok = 0;
  } else if (need > 0) {
    const int top = atomicSub(&s.counters[kCtrFreeTop], need);
    if (top - need < 0 || top > s.num_blocks) {
      atomicAdd(&s.counters[kCtrFreeTop], need);
      atomicOr(&s.counters[kCtrStatus], kDevOutOfBlocks);
      ok = 0;
    } else {
      int32_t* row = s.block_table + (size_t)b * s.max_bps;
      for (int j = 0; j < need; ++j) row[old_pages + j] = s.free_stack[top - 1 - j];
    }
  }
  if (ok) {
    s.seq_slots[b] = new_slots;
    s.seq_pos[b] = pos + n_new;
  }
  s.plan[2 * b] = ok ? slots : -1;
  s.plan[2 * b + 1] = pos;
}

template <int BITS>
__global__ void __launch_bounds__(512) append_rows_kernel(DevState s, int seq_begin, int n_new,
                                                          const uint16_t* __restrict__ kin,
                                                          const uint16_t* __restrict__ vin) {
  const int bl = blockIdx.y;
  const int b = seq_begin + bl;
  const int slots = s.plan[2 * b];
  if (slots < 0) return;
  const int pos = s.plan[2 * b + 1];
  int lo, hi;
  pool_range(pos, n_new, s.ring, &lo, &hi);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int hkv = s.hkv;
  const int W = s.ring;
  const int t0 = blockIdx.x * kBulkTokens;
  const int nt = min(kBulkTokens, n_new - t0);
  for (int row = warp; row < nt * hkv * 2; row += nwarps) {
    const int kv = row & 1;
    const int h = (row >> 1) % hkv;
    const int i = t0 + (row >> 1) / hkv;
    const uint16_t* src = (kv ? vin : kin) + (((size_t)bl * hkv + h) * n_new + i) * kHeadDim;
    const uint2 raw = *reinterpret_cast<const uint2*>(src + lane * 4);
    const int p = pos + i;
    if (p < kSinks) {
      uint16_t* dst = (kv ? s.sink_v : s.sink_k) + (((size_t)b * hkv + h) * kSinks + p) * kHeadDim;
      *reinterpret_cast<uint2*>(dst + lane * 4) = raw;
      if (kv == 0 && lane == 0) s.sink_score[((size_t)b * hkv + h) * kSinks + p] = 0.0f;
    } else if (p < hi) {
      quantize_row<BITS>(s, b, h, kv, slots + (p - lo), p, 0.0f, raw, lane);
    } else {
      const size_t ridx = ((size_t)b * hkv + h) * W + (p - kSinks) % W;
      uint16_t* dst = (kv ? s.ring_v : s.ring_k) + ridx * kHeadDim;
      *reinterpret_cast<uint2*>(dst + lane * 4) = raw;
      if (kv == 0 && lane == 0) s.ring_score[ridx] = 0.0f;
    }
  }
}

__global__ void fill_free_stack_kernel(int32_t* stack, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) stack[i] = n - 1 - i;
}

}  // namespace

cudaError_t launch_append_bulk(const DevState& s, int seq_begin, int batch, int n_new, const uint16_t* k,
                               const uint16_t* v, cudaStream_t st) {
  append_alloc_kernel<<<(batch + 127) / 128, 128, 0, st>>>(s, seq_begin, batch, n_new);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 grid((n_new + kBulkTokens - 1) / kBulkTokens, batch);
  if (s.bits == 8)
    append_rows_kernel<8><<<grid, 512, 0, st>>>(s, seq_begin, n_new, k, v);
  else
    append_rows_kernel<4><<<grid, 512, 0, st>>>(s, seq_begin, n_new, k, v);
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
