// Prefill: the causal attention of a fresh prompt over itself and the H2O
// scores it gives (Technical Report section 3.4: a token's score is the sum,
// over the query rows of the attention matrix, of its probabilities; the
// eviction-and-reuse survey page's section 3.3: its cumulative attention from
// the later tokens).  The prompt attends with its exact bf16 values; its
// tokens are stored quantised (or in the bf16 window) by the append that runs
// first, and the scores initialise the decode steps' H2O accumulation.
//
// Two kernels: the forward on tcgen05 (kvc_prefill_tc.cu: the bf16 output
// and each query row's (max, sum)), then the scores here, on mma.sync
// m16n8k16 with bf16 operands and fp32 accumulation (the query and key bits
// multiply exactly):
//
// prefill_scores_kernel, one 128-thread CTA per (64-key tile, KV head,
// sequence): the K tile stays in shared memory while the CTA walks every
// query tile at or after it of every query head of the group (Q tiles double
// buffered), recomputes S (the same exact products, summed in fp32), turns it into
// probabilities with the forward's row statistics, and sums them over the
// query rows; the column sums land in the tokens' score slots (sinks, pool
// or bf16 window).
//
// A prompt over sequences that already hold context (kvc_prefill_context)
// attends to the compressed cache instead (kvc_context.cu).
#include <cuda_bf16.h>

#include "kvc_device.h"
#include "kvc_internal.h"

namespace kvc {
namespace {

using namespace dev;

constexpr int kPfThreads = 128;
constexpr int kPfTile = 64;
constexpr int kPfRow = kHeadDim + 8;  // bf16 per staged row (272 bytes)
typedef uint16_t PfTile[kPfTile][kPfRow];

struct PfScoreSmem {
  PfTile k;
  PfTile q[2];
  float cs[kPfThreads / 32][kPfTile];
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src));
}

__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }

template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Copy `valid` rows of 128 bf16 (row stride 128 in global) into a staged
// tile; rows past `valid` are zeroed.
__device__ __forceinline__ void load_tile(PfTile& dst, const uint16_t* src, int valid) {
  for (int i = threadIdx.x; i < kPfTile * (kHeadDim / 8); i += kPfThreads) {
    const int r = i / (kHeadDim / 8), ch = i % (kHeadDim / 8);
    if (r < valid)
      cp_async16(smem_addr(&dst[r][ch * 8]), src + (size_t)r * kHeadDim + ch * 8);
    else
      *reinterpret_cast<uint4*>(&dst[r][ch * 8]) = make_uint4(0u, 0u, 0u, 0u);
  }
}

__device__ __forceinline__ void ldsm_x4(uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t& a3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
               : "r"(smem_addr(p)));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Q fragments (A operand) of this warp's 16 rows, all 8 k-steps.
__device__ __forceinline__ void load_q_frags(const PfTile& sq, int warp, int lane, uint32_t (&qa)[8][4]) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    ldsm_x4(qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], &sq[16 * warp + (lane & 15)][16 * kk + (lane >> 4) * 8]);
}

// S (16 x 64) = Q K^T for this warp: sc[nt][e], rows lane/4 (+8), keys
// 8 nt + 2 (lane % 4) (+1).
__device__ __forceinline__ void qk_tile(const uint32_t (&qa)[8][4], const PfTile& sk, int lane, float (&sc)[8][4]) {
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.0f;
#pragma unroll
    for (int kp = 0; kp < 4; ++kp) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(b0, b1, b2, b3, &sk[8 * nt + (lane & 7)][32 * kp + (lane >> 3) * 8]);
      mma_bf16(sc[nt], qa[2 * kp][0], qa[2 * kp][1], qa[2 * kp][2], qa[2 * kp][3], b0, b1);
      mma_bf16(sc[nt], qa[2 * kp + 1][0], qa[2 * kp + 1][1], qa[2 * kp + 1][2], qa[2 * kp + 1][3], b2, b3);
    }
  }
}

__global__ void __launch_bounds__(kPfThreads) prefill_scores_kernel(DevState s, int n,
                                                                    const uint16_t* __restrict__ q,
                                                                    const uint16_t* __restrict__ k,
                                                                    const float* __restrict__ stats,
                                                                    float qk_scale_log2, int seq_begin) {
  extern __shared__ __align__(16) uint8_t pf_smem[];
  PfScoreSmem& sm = *reinterpret_cast<PfScoreSmem*>(pf_smem);
  const int kt = blockIdx.x, h = blockIdx.y, bl = blockIdx.z;
  const int b = seq_begin + bl;
  const int G = s.group;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = lane >> 2, c = lane & 3;
  const int k0 = kt * kPfTile;
  const int n_qt = (n + kPfTile - 1) / kPfTile;
  const int per_head = n_qt - kt;  // query tiles kt .. n_qt - 1
  const int iters = G * per_head;

  load_tile(sm.k, k + (((size_t)bl * s.hkv + h) * n + k0) * kHeadDim, min(kPfTile, n - k0));
  auto q_tile = [&](int it, PfTile& dst) {
    const int g = it / per_head, qt = kt + it % per_head;
    const size_t qrow0 = ((size_t)bl * s.hq + h * G + g) * n;
    load_tile(dst, q + (qrow0 + (size_t)qt * kPfTile) * kHeadDim, min(kPfTile, n - qt * kPfTile));
  };
  q_tile(0, sm.q[0]);
  cp_commit();

  float cs[8][2];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) cs[nt][0] = cs[nt][1] = 0.0f;

  for (int it = 0; it < iters; ++it) {
    if (it + 1 < iters) q_tile(it + 1, sm.q[(it + 1) & 1]);
    cp_commit();
    cp_wait<1>();
    __syncthreads();
    const int g = it / per_head, qt = kt + it % per_head;
    const size_t qrow0 = ((size_t)bl * s.hq + h * G + g) * n;
    uint32_t qa[8][4];
    load_q_frags(sm.q[it & 1], warp, lane, qa);
    float sc[8][4];
    qk_tile(qa, sm.k, lane, sc);
    // the forward kernel's row statistics of this warp's two query rows
    float rm[2], rinv[2];
    int qi[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      qi[rr] = qt * kPfTile + 16 * warp + r + 8 * rr;
      float2 st = make_float2(0.0f, 1.0f);
      if (qi[rr] < n) st = *reinterpret_cast<const float2*>(stats + (qrow0 + qi[rr]) * 2);
      rm[rr] = st.x;
      rinv[rr] = 1.0f / st.y;
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int ki = k0 + 8 * nt + 2 * c + (e & 1);
        const int rr = e >> 1;
        const bool ok = ki <= qi[rr] && ki < n && qi[rr] < n;
        const float p = ok ? fast_exp2(sc[nt][e] * qk_scale_log2 - rm[rr]) * rinv[rr] : 0.0f;
        cs[nt][e & 1] += p;
      }
    }
    __syncthreads();  // the next iteration's copies overwrite this Q buffer
  }
  cp_wait<0>();

  // sum over the warp's rows (lanes with the same lane % 4), then the warps
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      float v = cs[nt][x];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      if (r == 0) sm.cs[warp][8 * nt + 2 * c + x] = v;
    }
  }
  __syncthreads();
  const int t = threadIdx.x;
  if (t < kPfTile && k0 + t < n) {
    float v = 0.0f;
#pragma unroll
    for (int w = 0; w < kPfThreads / 32; ++w) v += sm.cs[w][t];
    const int p = k0 + t;
    int lo, hi;
    pool_range(0, n, s.ring, &lo, &hi);
    if (p < kSinks) {
      s.sink_score[((size_t)b * s.hkv + h) * kSinks + p] = v;
    } else if (p < hi) {
      const int slot = p - lo;
      const int blk = s.block_table[(size_t)b * s.max_bps + slot / kPage];
      if ((unsigned)blk < (unsigned)s.num_blocks)
        s.score[((size_t)blk * s.hkv + h) * kPage + slot % kPage] = v;
      else
        atomicOr(&s.counters[kCtrStatus], kDevBadBlockId);
    } else {
      s.ring_score[((size_t)b * s.hkv + h) * s.ring + (p - kSinks) % s.ring] = v;
    }
  }
}

}  // namespace

int prefill_scores_smem_bytes() { return (int)sizeof(PfScoreSmem); }

cudaError_t launch_prefill(const DevState& s, int seq_begin, int batch, int n, const uint16_t* q, const uint16_t* k,
                           const uint16_t* v, uint16_t* out, float* stats, float qk_scale_log2, bool scores,
                           cudaStream_t st, cudaEvent_t trace_start, cudaEvent_t trace_stop) {
  static int done_sc[64] = {0};
  cudaError_t e = trace_start ? cudaEventRecord(trace_start, st) : cudaSuccess;
  if (e != cudaSuccess) return e;
  e = launch_prefill_fwd_tc(s, batch, n, q, k, v, out, stats, qk_scale_log2, st);
  if (e == cudaSuccess && trace_stop) e = cudaEventRecord(trace_stop, st);
  if (e != cudaSuccess || !scores) return e;
  const int tiles = (n + kPfTile - 1) / kPfTile;
  e = opt_in_smem(reinterpret_cast<const void*>(prefill_scores_kernel), prefill_scores_smem_bytes(), done_sc);
  if (e != cudaSuccess) return e;
  prefill_scores_kernel<<<dim3(tiles, s.hkv, batch), kPfThreads, prefill_scores_smem_bytes(), st>>>(
      s, n, q, k, stats, qk_scale_log2, seq_begin);
  return cudaGetLastError();
}

}  // namespace kvc
