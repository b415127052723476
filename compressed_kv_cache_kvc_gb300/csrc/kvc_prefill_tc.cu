// Prefill forward on the fifth-generation tensor cores: the causal attention
// of a fresh prompt over itself (Technical Report section 1.1), with S = Q K^T
// and O = P V by tcgen05.mma (fp32 accumulators in tensor memory).  Outputs
// and row statistics (m, l) as the decode kernels define them; the H2O
// scores come from prefill_scores_kernel (kvc_prefill.cu), which uses these
// statistics.
//
// One 256-thread CTA per (128-query tile, query head, sequence); threads t
// and t + 128 own query row t (TMEM lane t), the first S columns [0, 32) and
// O columns [0, 64), the second the other halves; they agree on the row
// maximum through shared memory.  Per 64-key tile (up to the diagonal):
//   * K rows by cp.async into the operand layout (K-major, no swizzle:
//     8-row x 16-byte core matrices), V rows into a staging tile (16-byte
//     chunks XOR-swizzled by row), both double-buffered: tile j + 1's copies
//     run while tile j is computed; V is transposed by ldmatrix.trans into a
//     dims x keys operand and converted to fp16 on the way;
//   * one thread issues S = Q K^T (M 128, N 64, 8 MMAs of K 16, bf16: exact
//     products) into TMEM columns [0, 64);
//   * each thread reads its half row of S (tcgen05.ld), masks (only tiles
//     that cross the diagonal or the end of the prompt), and runs the
//     online softmax in the log2 domain with a lazy maximum (O in TMEM is
//     rescaled only when the row maximum grows by more than 8);
//   * P in fp16 (11 significant bits; p <= 2^8 by the lazy maximum) over the
//     K buffer S has finished with, and one thread issues O += P V (M 128,
//     N 128, K 64, fp16 operands) into columns [128, 256).  A bf16 P alone
//     missed the output tolerance on rows that see few keys; P in two bf16
//     parts (hi + lo) met it at two MMAs per tile, 12-15 % slower overall.
//     V entries beyond fp16's range (|v| >= 65536, or not finite) saturate
//     to +-65504 and set KVC_DEV_PREFILL_RANGE.
// Every mbarrier wait is bounded; a wait that runs out sets
// KVC_DEV_WAIT_TIMEOUT, and the CTA stops after freeing its tensor memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kvc_device.h"
#include "kvc_internal.h"

namespace kvc {
namespace {

using namespace dev;

constexpr int kTcThreads = 256;      // two threads per query row (TMEM lane)
constexpr int kTcQ = 128;            // queries per CTA (the MMAs' M)
constexpr int kTcKeys = 64;          // keys per tile
constexpr float kTcLazy = 8.0f;      // log2 units the running maximum may lag
constexpr uint32_t kTcCols = 256;    // TMEM columns: S [0, 64), O [128, 256)
constexpr uint32_t kTcO = 128;
constexpr int kTcWaitLimit = 1 << 22;

constexpr int kTileBytes = kTcKeys * kHeadDim * 2;          // 16 KB
constexpr int kOffQ = 0;                                     // 32 KB: Q, operand layout
constexpr int kOffK = kOffQ + kTcQ * kHeadDim * 2;           // 2 x 16 KB: K, then P (operand layout)
constexpr int kOffV = kOffK + 2 * kTileBytes;                // 2 x 16 KB: staged V
constexpr int kOffVt = kOffV + 2 * kTileBytes;               // 16 KB: V^T in fp16, operand layout
constexpr int kOffBar = kOffVt + kTileBytes;                 // mbarrier, TMEM base
constexpr int kTcSmem = kOffBar + 16;                        // two CTAs per SM

// Staged V: row r (a key) of 256 bytes, its 16-byte chunk c at c ^ (r % 8),
// so the 8 rows an ldmatrix reads together lie on different banks.
__device__ __forceinline__ int vstage_off(int r, int c) { return r * 256 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Byte offset of 16-byte chunk c (elements 8c .. 8c + 7) of row r in the
// operand layout of a tile with `kch` chunks per row: core matrices of 8 rows
// x 16 bytes, row groups kch * 128 bytes apart, chunks 128 bytes apart.
__device__ __forceinline__ int core_off(int r, int c, int kch) { return ((r >> 3) * kch + c) * 128 + (r & 7) * 16; }

// Shared-memory operand descriptor: K-major, no swizzle; leading byte offset
// (between the two core matrices of a K step) 128, stride byte offset
// `sbo` (between 8-row groups); descriptor version 1.
__device__ __forceinline__ uint64_t op_desc(uint32_t addr, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) |
         ((uint64_t)1 << 46);
}

// fp16 bits of 65504, its largest finite value.  bf16 magnitudes from 65536
// up saturate to it; 65280, the bf16 value below, converts exactly.
constexpr uint32_t kF16Max = 0x7BFFu;

// (lo, hi) to fp16x2, round to nearest, out-of-range values saturated to
// +-65504 (NaN stays NaN).
__device__ __forceinline__ uint32_t f16x2_sat(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Instruction descriptor of kind::f16: f32 accumulator, A and B both bf16
// (`bf16`) or both fp16, both K-major, N / 8 at bit 17, M / 16 at bit 24.
__device__ __forceinline__ uint32_t instr_desc(int m, int n, bool bf16) {
  const uint32_t ab = bf16 ? ((1u << 7) | (1u << 10)) : 0u;
  return (1u << 4) | ab | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t dtmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(dtmem),
      "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)acc));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Bounded wait for the mbarrier's phase `parity`; true when it completed.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity) {
  uint32_t done = 0;
  for (int it = 0; it < kTcWaitLimit && !done; ++it)
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
  return done != 0;
}

__device__ __forceinline__ void ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])));
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Shared-memory writes by threads, then work for the tensor cores (async proxy).
__device__ __forceinline__ void publish_to_mma() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__global__ void __launch_bounds__(kTcThreads, 2) prefill_fwd_tc_kernel(DevState s, int n,
                                                                      const uint16_t* __restrict__ q,
                                                                      const uint16_t* __restrict__ k,
                                                                      const uint16_t* __restrict__ v,
                                                                      uint16_t* __restrict__ out,
                                                                      float* __restrict__ stats, float qk_scale_log2) {
  extern __shared__ __align__(1024) uint8_t tc_smem[];
  uint8_t* sq = tc_smem + kOffQ;
  uint8_t* svt = tc_smem + kOffVt;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(tc_smem + kOffBar);
  uint32_t* tbase = reinterpret_cast<uint32_t*>(tc_smem + kOffBar + 8);
  const uint32_t bar = saddr(mbar);

  // the longest (last) query tiles first
  const int qt = gridDim.x - 1 - blockIdx.x, hqi = blockIdx.y, bl = blockIdx.z;
  const int hkvi = hqi / s.group;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // thread (half h, row r): query row r, S columns [32 h, 32 h + 32), O
  // columns [64 h, 64 h + 64); warps w and w + 4 share TMEM lanes 32 (w % 4) ..
  const int half = tid >> 7, r = tid & (kTcQ - 1);
  const size_t qrow0 = ((size_t)bl * s.hq + hqi) * n;
  const uint16_t* kb = k + ((size_t)bl * s.hkv + hkvi) * n * kHeadDim;
  const uint16_t* vb = v + ((size_t)bl * s.hkv + hkvi) * n * kHeadDim;
  const int q0 = qt * kTcQ;
  const int qi = q0 + r;  // this thread's query row
  const int n_kt = min((q0 + kTcQ - 1) / kTcKeys + 1, (n + kTcKeys - 1) / kTcKeys);

  // Q tile into the operand layout (rows past n zero); 8 consecutive threads
  // fill one core matrix (8 rows of one 16-byte chunk: 128 contiguous bytes)
  for (int i = tid; i < kTcQ * (kHeadDim / 8); i += kTcThreads) {
    const int rr = (i & 7) | ((i >> 7) << 3), c = (i >> 3) & 15;
    uint8_t* d = sq + core_off(rr, c, kHeadDim / 8);
    if (q0 + rr < n)
      cp16(saddr(d), q + (qrow0 + q0 + rr) * kHeadDim + 8 * c);
    else
      *reinterpret_cast<uint4*>(d) = make_uint4(0u, 0u, 0u, 0u);
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tbase)),
                 "r"(kTcCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tbase;
  const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);  // this warp's lanes

  const uint32_t id_s = instr_desc(kTcQ, kTcKeys, true);
  const uint32_t id_o = instr_desc(kTcQ, kHeadDim, false);
  float m = kNegBig, l = 0.0f;  // l: the sum over this thread's columns
  uint32_t phase = 0;
  bool ok = true;
  __half2 vmax = __floats2half2_rn(0.0f, 0.0f);  // largest |V| in fp16 (NaN kept)

  // copies of key tile jt into buffers jt % 2 (rows past n zero): K in the
  // operand layout (8 consecutive threads per core matrix), V in the staging
  // layout (16 consecutive threads per row)
  auto load_kv = [&](int jt) {
    const int k0 = jt * kTcKeys;
    uint8_t* dkb = tc_smem + kOffK + (jt & 1) * kTileBytes;
    uint8_t* dvb = tc_smem + kOffV + (jt & 1) * kTileBytes;
#pragma unroll
    for (int it = 0; it < kTcKeys * (kHeadDim / 8) / kTcThreads; ++it) {
      const int i = tid + it * kTcThreads;
      const int rk = (i & 7) | ((i >> 7) << 3), ck = (i >> 3) & 15;
      const int rv = i >> 4, cv = i & 15;
      uint8_t* dk = dkb + core_off(rk, ck, kHeadDim / 8);
      uint8_t* dv = dvb + vstage_off(rv, cv);
      if (k0 + rk < n)
        cp16(saddr(dk), kb + (size_t)(k0 + rk) * kHeadDim + 8 * ck);
      else
        *reinterpret_cast<uint4*>(dk) = make_uint4(0u, 0u, 0u, 0u);
      if (k0 + rv < n)
        cp16(saddr(dv), vb + (size_t)(k0 + rv) * kHeadDim + 8 * cv);
      else
        *reinterpret_cast<uint4*>(dv) = make_uint4(0u, 0u, 0u, 0u);
    }
  };
  load_kv(0);  // one copy group with Q
  asm volatile("cp.async.commit_group;" ::: "memory");

  for (int j = 0; j < n_kt && ok; ++j) {
    const int k0 = j * kTcKeys;
    uint8_t* sk = tc_smem + kOffK + (j & 1) * kTileBytes;
    uint8_t* sv = tc_smem + kOffV + (j & 1) * kTileBytes;
    // the next tile's copies into the other buffers (free: the previous
    // tile's MMAs, which read them as P, completed), then this tile's wait
    if (j + 1 < n_kt) load_kv(j + 1);
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 1;" ::: "memory");
    __syncthreads();
    // V^T (dims x keys) in fp16 in the operand layout: the 8 x 8 block (key
    // group kg, dim group dg) of V transposed is core matrix (dg, kg) of V^T;
    // warp w transposes key group w
#pragma unroll
    for (int bi = 0; bi < 4; ++bi) {
      const int kg = warp, dg = 4 * bi;  // 4 blocks per ldmatrix: dims 8 (dg .. dg + 3)
      const int mi = lane >> 3, rr = lane & 7;
      uint32_t t0, t1, t2, t3;
      asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                   : "=r"(t0), "=r"(t1), "=r"(t2), "=r"(t3)
                   : "r"(saddr(sv + vstage_off(8 * kg + rr, dg + mi))));
      const uint32_t tv[4] = {t0, t1, t2, t3};
#pragma unroll
      for (int mm = 0; mm < 4; ++mm) {
        const uint32_t hv = f16x2_sat(bf16f(tv[mm] & 0xFFFFu), bf16f(tv[mm] >> 16));
        vmax = __hmax2_nan(vmax, __habs2(*reinterpret_cast<const __half2*>(&hv)));
        *reinterpret_cast<uint32_t*>(svt + core_off(8 * (dg + mm) + (lane >> 2), kg, kTcKeys / 8) +
                                     4 * (lane & 3)) = hv;
      }
    }
    publish_to_mma();
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < kHeadDim / 16; ++ks)
        mma_f16(tmem, op_desc(saddr(sq) + ks * 256, (kHeadDim / 8) * 128),
                op_desc(saddr(sk) + ks * 256, (kHeadDim / 8) * 128), id_s, ks > 0);
      mma_commit(bar);
    }
    ok = __syncthreads_and(bar_wait(bar, phase));
    phase ^= 1u;
    if (!ok) break;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

    // this thread's 32 raw logits; only tiles that cross the diagonal or
    // the end of the prompt are masked (the test is the same for the CTA)
    float x[kTcKeys / 2];
    ld16(trow + 32 * half, *reinterpret_cast<float(*)[16]>(&x[0]));
    ld16(trow + 32 * half + 16, *reinterpret_cast<float(*)[16]>(&x[16]));
    if (k0 + kTcKeys - 1 > q0 || k0 + kTcKeys > n) {
#pragma unroll
      for (int i = 0; i < kTcKeys / 2; ++i) {
        const int ki = k0 + 32 * half + i;
        if (!(ki <= qi && ki < n)) x[i] = -INFINITY;
      }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < kTcKeys / 2; ++i) mx = fmaxf(mx, x[i]);
    // the row maximum from the two halves, through this tile's V staging
    // (transposed already; the next copies into it start after two more
    // barriers)
    float* red = reinterpret_cast<float*>(sv);
    red[half * kTcQ + r] = mx;
    __syncthreads();
    mx = fmaxf(mx, red[(half ^ 1) * kTcQ + r]) * qk_scale_log2;  // scale > 0: the max commutes
    // the row maximum moved: rescale the sum and (after the first tile) O.
    // TMEM loads and stores are warp-collective: the warp rescales when any
    // of its rows must, the others by 1; both halves decide alike
    const bool grow = mx > m + kTcLazy;
    const float alpha = grow ? fast_exp2(m - mx) : 1.0f;
    if (grow) {
      l *= alpha;
      m = mx;
    }
    if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll 1
      for (int c0 = 0; c0 < kHeadDim / 2; c0 += 16) {
        float t[16];
        ld16(trow + kTcO + 64 * half + c0, t);
#pragma unroll
        for (int i = 0; i < 16; ++i) t[i] *= alpha;
        st16(trow + kTcO + 64 * half + c0, t);
      }
    }
    // P in fp16 over K of this tile (the sum adds the unrounded p, as the
    // decode kernels do)
    const float nm = -m;
#pragma unroll
    for (int c = 0; c < kTcKeys / 16; ++c) {
      uint32_t hw[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p0 = fast_exp2(fmaf(x[8 * c + 2 * e], qk_scale_log2, nm));
        const float p1 = fast_exp2(fmaf(x[8 * c + 2 * e + 1], qk_scale_log2, nm));
        l += p0 + p1;
        const __half2 h = __floats2half2_rn(p0, p1);
        hw[e] = *reinterpret_cast<const uint32_t*>(&h);
      }
      *reinterpret_cast<uint4*>(sk + core_off(r, 4 * half + c, kTcKeys / 8)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    }
    publish_to_mma();
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < kTcKeys / 16; ++ks)
        mma_f16(tmem + kTcO, op_desc(saddr(sk) + ks * 256, (kTcKeys / 8) * 128),
                op_desc(saddr(svt) + ks * 256, (kTcKeys / 8) * 128), id_o, j > 0 || ks > 0);
      mma_commit(bar);
    }
    ok = __syncthreads_and(bar_wait(bar, phase));
    phase ^= 1u;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  }

  if (ok) {
    // the row's sum from the two halves (V^T is free: the MMAs completed)
    float* red = reinterpret_cast<float*>(svt);
    red[half * kTcQ + r] = l;
    __syncthreads();
    l += red[(half ^ 1) * kTcQ + r];
    // O / l to bf16, and the row's (max, sum); every lane reads (the TMEM
    // load is warp-collective), rows past n store nothing
    const bool row_ok = qi < n;
    const float inv = row_ok ? 1.0f / l : 0.0f;
    uint16_t* orow = out + (qrow0 + (row_ok ? qi : 0)) * kHeadDim + 64 * half;
#pragma unroll 1
    for (int c0 = 0; c0 < kHeadDim / 2; c0 += 16) {
      float t[16];
      ld16(trow + kTcO + 64 * half + c0, t);
      uint32_t w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const __nv_bfloat162 pr = __floats2bfloat162_rn(t[2 * e] * inv, t[2 * e + 1] * inv);
        w[e] = *reinterpret_cast<const uint32_t*>(&pr);
      }
      if (row_ok) {
        *reinterpret_cast<uint4*>(orow + c0) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(orow + c0 + 8) = make_uint4(w[4], w[5], w[6], w[7]);
      }
    }
    if (row_ok && half == 0) *reinterpret_cast<float2*>(stats + (qrow0 + qi) * 2) = make_float2(m, l);
  } else {
    if (tid == 0) atomicOr(&s.counters[kCtrStatus], kDevWaitTimeout);
    // a last bounded wait for the MMAs whose completion did not come (the
    // phase was flipped after the failed wait) before the columns go back
    bar_wait(bar, phase ^ 1u);
  }
  // a saturated V entry reads 65504 in fp16, which no bf16 value converts to
  const uint32_t vmb = *reinterpret_cast<const uint32_t*>(&vmax);
  if ((vmb & 0x7FFFu) >= kF16Max || ((vmb >> 16) & 0x7FFFu) >= kF16Max)
    atomicOr(&s.counters[kCtrStatus], kDevPrefillRange);
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcCols));
}

}  // namespace

int prefill_fwd_tc_smem_bytes() { return kTcSmem; }

cudaError_t launch_prefill_fwd_tc(const DevState& s, int batch, int n, const uint16_t* q, const uint16_t* k,
                                  const uint16_t* v, uint16_t* out, float* stats, float qk_scale_log2,
                                  cudaStream_t st) {
  static int done[64] = {0};
  const cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(prefill_fwd_tc_kernel), kTcSmem, done);
  if (e != cudaSuccess) return e;
  const int tiles = (n + kTcQ - 1) / kTcQ;
  prefill_fwd_tc_kernel<<<dim3(tiles, s.hq, batch), kTcThreads, kTcSmem, st>>>(s, n, q, k, v, out, stats,
                                                                               qk_scale_log2);
  return cudaGetLastError();
}

}  // namespace kvc
