// Decode attention over the bf16 window of hybrid precision ("KV Cache
// optimization techniques" section 1.3, HybridPrecisionKVCache: recent tokens
// kept at 16 bits).  The tokens of the last W positions of a sequence live in
// a bf16 ring per (sequence, KV head); this kernel attends the query heads of
// a KV head to them with their exact values and leaves, per chunk of 64 ring
// slots, one partial (m, l, o) that the merge folds in with the split-K
// partials of the quantised pool and the sinks, plus the log2-domain logits
// that the H2O score pass reads.
//
// One 128-thread CTA per (chunk, KV head, sequence).  The chunk's K and V rows
// are copied to shared memory with cp.async (rows padded to 272 bytes, so the
// ldmatrix row addresses fall in different banks).  QK^T: each warp takes 16
// slots and runs mma.sync m16n8k16 with bf16 operands (slots on M, query
// heads on N, padded to 8): the query's own bf16 bits and the stored bf16
// keys multiply exactly, the sums accumulate in fp32.  PV: mma.sync again,
// head dimensions on M (32 per warp), query heads on N, slots on K, with the
// probabilities split into two bf16 parts (16 significant bits in all).
#include <cuda_bf16.h>

#include "kvc_device.h"
#include "kvc_internal.h"

namespace kvc {
namespace {

using namespace dev;

constexpr int kRingThreads = 128;
constexpr int kRowPad = kHeadDim + 8;  // bf16 per staged row (272 bytes)

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src));
}

__global__ void __launch_bounds__(kRingThreads) attn_ring_kernel(DevState s, int seq_begin,
                                                                 const uint16_t* __restrict__ q,
                                                                 float qk_scale_log2, AttnWork w) {
  __shared__ __align__(16) uint16_t sk[kRingChunk][kRowPad];
  __shared__ __align__(16) uint16_t sv[kRingChunk][kRowPad];
  __shared__ __align__(16) float sp[kRingChunk][kMaxGroup];  // logits, then probabilities
  __shared__ float sm_m[kMaxGroup], sm_l[kMaxGroup];
  const int chunk = blockIdx.x;
  const int h = blockIdx.y;
  const int bl = blockIdx.z;
  const int b = seq_begin + bl;
  const int hkv = s.hkv;
  const int G = s.group;
  const int W = s.ring;
  const int nr = ring_count(s.seq_pos[b], W);
  const int slot0 = chunk * kRingChunk;
  const int n_here = min(kRingChunk, nr - slot0);
  if (n_here <= 0) return;  // the merge reads only the chunks that hold tokens
  const int pair = bl * hkv + h;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // ---- stage the chunk's rows: K, then V as a second group that lands
  // while QK^T and the softmax run
  const size_t row0 = ((size_t)b * hkv + h) * W + slot0;
  for (int i = threadIdx.x; i < n_here * (kHeadDim / 8); i += kRingThreads) {
    const int row = i / (kHeadDim / 8), ch = i % (kHeadDim / 8);
    cp_async16(smem_addr(&sk[row][ch * 8]), s.ring_k + (row0 + row) * kHeadDim + ch * 8);
  }
  asm volatile("cp.async.commit_group;\n" ::);
  for (int i = threadIdx.x; i < n_here * (kHeadDim / 8); i += kRingThreads) {
    const int row = i / (kHeadDim / 8), ch = i % (kHeadDim / 8);
    cp_async16(smem_addr(&sv[row][ch * 8]), s.ring_v + (row0 + row) * kHeadDim + ch * 8);
  }
  asm volatile("cp.async.commit_group;\n" ::);

  // ---- query fragments (B operand, k16 x n8): lane holds query head n = lane / 4,
  // dims 2(lane % 4) + {0, 1} and + 8 of every 16-dim step; heads >= G are 0
  const int n = lane >> 2, c = lane & 3;
  uint32_t bq[8][2];
  {
    const uint32_t* qr = reinterpret_cast<const uint32_t*>(q + ((size_t)bl * s.hq + h * G + n) * kHeadDim);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      bq[kk][0] = n < G ? qr[8 * kk + c] : 0u;
      bq[kk][1] = n < G ? qr[8 * kk + 4 + c] : 0u;
    }
  }
  asm volatile("cp.async.wait_group 1;\n" ::: "memory");  // K is in
  __syncthreads();

  // ---- logits of 16 slots per warp
  if (16 * warp < n_here) {
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const uint32_t abase = smem_addr(&sk[16 * warp + (lane & 15)][(lane >> 4) * 8]);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t a0, a1, a2, a3;
      asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                   : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                   : "r"(abase + kk * 32));
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
          "{%0, %1, %2, %3};\n"
          : "+f"(acc[0]), "+f"(acc[1]), "+f"(acc[2]), "+f"(acc[3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(bq[kk][0]), "r"(bq[kk][1]));
    }
    // C fragment: slots 16 warp + lane / 4 (+ 8), query heads 2 (lane % 4) + {0, 1}
    const int r = lane >> 2;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int row = 16 * warp + r + (e >= 2 ? 8 : 0);
      const int g = 2 * c + (e & 1);
      const bool ok = row < n_here && g < G;
      const float lg = ok ? acc[e] * qk_scale_log2 : -INFINITY;
      sp[row][g] = lg;
      if (ok) w.ring_lg[((size_t)pair * G + g) * W + slot0 + row] = lg;
    }
  }
  __syncthreads();

  // ---- per query head: max and sum of the chunk (warp g % 4 takes head g)
  for (int g = warp; g < G; g += kRingThreads / 32) {
    float m = kNegBig;
    for (int t = lane; t < n_here; t += 32) m = fmaxf(m, sp[t][g]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.0f;
    for (int t = lane; t < n_here; t += 32) l += fast_exp2(sp[t][g] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) {
      sm_m[g] = m;
      sm_l[g] = l;
    }
  }
  __syncthreads();
  // probabilities of the k-steps' slots (0 past n_here) and zero V rows past
  // n_here in the last k-step: their probability is 0, but 0 times stale
  // shared memory could be NaN
  const int kt = (n_here + 15) >> 4;  // 16-slot k-steps of PV
  for (int i = threadIdx.x; i < 16 * kt * kMaxGroup; i += kRingThreads) {
    const int t = i / kMaxGroup, g = i % kMaxGroup;
    sp[t][g] = (t < n_here && g < G) ? fast_exp2(sp[t][g] - sm_m[g]) : 0.0f;
  }
  for (int i = threadIdx.x; i < (16 * kt - n_here) * (kHeadDim / 8); i += kRingThreads)
    *reinterpret_cast<uint4*>(&sv[n_here + i / (kHeadDim / 8)][(i % (kHeadDim / 8)) * 8]) = make_uint4(0u, 0u, 0u, 0u);
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");  // V is in
  __syncthreads();

  // ---- O^T (head dims x query heads) = V^T . P on the tensor cores: warp w
  // takes dims 32w .. 32w + 31 (two M tiles), the slots are K.  V^T comes
  // from the staged rows by ldmatrix.trans; P enters as two bf16 parts, hi =
  // bf16(p) and lo = bf16(p - hi) (p - hi is exact in fp32), so the operand
  // carries 16 significant bits and the products are exact.
  float oc[2][4];
#pragma unroll
  for (int m = 0; m < 2; ++m) oc[m][0] = oc[m][1] = oc[m][2] = oc[m][3] = 0.0f;
  const int tr = (lane & 7) + ((lane >> 4) << 3);  // ldmatrix.trans row (slot) of this lane
  const int tc = ((lane >> 3) & 1) * 8;            // and column (dim) offset
  for (int kk = 0; kk < kt; ++kk) {
    uint32_t bh[2], bl[2];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int t = 16 * kk + 8 * half + 2 * c;
      const float p0 = sp[t][n], p1 = sp[t + 1][n];
      const __nv_bfloat162 hi = __floats2bfloat162_rn(p0, p1);
      const __nv_bfloat162 lo = __floats2bfloat162_rn(p0 - __low2float(hi), p1 - __high2float(hi));
      bh[half] = *reinterpret_cast<const uint32_t*>(&hi);
      bl[half] = *reinterpret_cast<const uint32_t*>(&lo);
    }
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      uint32_t a0, a1, a2, a3;
      asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                   : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                   : "r"(smem_addr(&sv[16 * kk + tr][32 * warp + 16 * m + tc])));
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
          "{%0, %1, %2, %3};\n"
          : "+f"(oc[m][0]), "+f"(oc[m][1]), "+f"(oc[m][2]), "+f"(oc[m][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(bh[0]), "r"(bh[1]));
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
          "{%0, %1, %2, %3};\n"
          : "+f"(oc[m][0]), "+f"(oc[m][1]), "+f"(oc[m][2]), "+f"(oc[m][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(bl[0]), "r"(bl[1]));
    }
  }
  // C fragment: dims 32w + 16m + lane / 4 (+ 8), query heads 2 (lane % 4) + {0, 1}
  const size_t pidx = (size_t)pair * w.ring_chunks + chunk;
#pragma unroll
  for (int m = 0; m < 2; ++m) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int d = 32 * warp + 16 * m + (lane >> 2) + (e >= 2 ? 8 : 0);
      const int g = 2 * c + (e & 1);
      if (g < G) w.ring_po[(pidx * G + g) * kHeadDim + d] = oc[m][e];
    }
  }
  const int d = threadIdx.x;
  if (d < G) {
    w.ring_pml[(pidx * G + d) * 2 + 0] = sm_m[d];
    w.ring_pml[(pidx * G + d) * 2 + 1] = sm_l[d];
  }
}

}  // namespace

cudaError_t launch_attention_ring(const DevState& s, int seq_begin, int batch, const uint16_t* q,
                                  float qk_scale_log2, const AttnWork& w, cudaStream_t st) {
  if (s.ring <= 0 || w.ring_chunks <= 0) return cudaSuccess;
  dim3 grid(w.ring_chunks, s.hkv, batch);
  attn_ring_kernel<<<grid, kRingThreads, 0, st>>>(s, seq_begin, q, qk_scale_log2, w);
  return cudaGetLastError();
}

}  // namespace kvc
