// Prefill on the fifth-generation tensor cores.  The forward: the causal
// attention of a fresh prompt over itself (Technical Report section 1.1), with
// S = Q K^T and O = P V by tcgen05.mma (fp32 accumulators in tensor memory),
// the outputs and row statistics (m, l) as the decode kernels define them.
// The H2O scores: prefill_scores_tc_kernel further down, from those
// statistics.
//
// One 448-thread CTA per (256-query block, query head, sequence), longest
// blocks first, warps with fixed roles:
//   * warpgroups 0 and 1 ("A" and "B") each own one 128-query tile; thread t
//     of a warpgroup owns query row t of its tile, TMEM lane t.  TMEM columns:
//     S_A [0, 64), S_B [64, 128), O_A [128, 256), O_B [256, 384), P_A
//     [384, 416), P_B [416, 448) (P in fp16, two per column);
//   * warpgroup 2 (the producer) brings both query tiles in by TMA (two
//     64-dim x 128-row boxes each, 128-byte swizzle; the S product reads them
//     in place) and 64-key tiles into a ring of three slots by TMA (one
//     thread issues the tensor copies, an mbarrier counts their bytes; rows
//     past the prompt read as zeros): K and V each as two 64 x 64 boxes
//     with the 128-byte swizzle; K is read in place by the MMA
//     (K-major, 128-byte swizzle), V is staged and the warpgroup transposes
//     it by ldmatrix.trans into a dims x keys operand in fp16 (K-major, no
//     swizzle, 8-row x 16-byte core matrices).  A slot is refilled once both
//     query tiles' P V products have read it;
//   * warps 12 and 13 issue the tensor-core products of query tiles A and B,
//     one thread each (one thread issues a product about every 100 cycles,
//     two threads together nearly twice as many): S(j + 1) = Q K(j + 1)^T
//     (M 128, N 64, bf16: exact products) as soon as the query tile has read
//     S(j), O += P V(j) (M 128, N 128, K 64, fp16, P read from tensor memory
//     as the A operand) as soon as it has written P(j).
// Per key tile j a query warpgroup waits for S(j), reads its S row
// (tcgen05.ld), masks (only tiles that cross the diagonal or the end of the
// prompt), runs the online softmax in the log2 domain with a lazy maximum (O
// is rescaled in TMEM only when the row maximum grows by more than 8), waits
// for P V(j - 1), and writes P in fp16 (11 significant bits; p <= 2^8 by the
// lazy maximum) into tensor memory.  The two query warpgroups run out of
// step, so one's softmax overlaps the other's products and the producer's
// copies overlap both.  A bf16 P alone missed the output tolerance on rows
// that see few keys.  V entries beyond fp16's range (|v| >= 65536, or not
// finite) saturate to +-65504 and set KVC_DEV_PREFILL_RANGE.
//
// Synchronisation: mbarriers (Q and K/V tiles landed, counted in bytes; S
// read and P written by the query warpgroups; slot full from the producer;
// slot empty and S / P V complete through tcgen05.commit) and named barriers
// inside a warpgroup.  Every mbarrier wait is bounded and also ends when
// another thread has given up;
// a wait that runs out sets KVC_DEV_WAIT_TIMEOUT, every role leaves its loop,
// the issuing thread waits (bounded) for its products in flight, and the
// CTA frees its tensor memory.
#include <cuda.h>  // CUtensorMap; the encoder comes through the runtime's driver entry point
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kvc_device.h"
#include "kvc_internal.h"

namespace kvc {
namespace {

using namespace dev;

constexpr int kWg = 128;                  // threads per warpgroup
constexpr int kTcThreads = 3 * kWg + 64;  // query tiles A and B, producer, two MMA warps
constexpr int kTcQ = 128;                 // queries per tile (the MMAs' M)
constexpr int kTcBlock = 2 * kTcQ;        // queries per CTA
constexpr int kTcKeys = 64;               // keys per tile
constexpr int kSlots = 3;                 // K / V^T ring
constexpr float kTcLazy = 8.0f;           // log2 units the running maximum may lag
constexpr uint32_t kTcCols = 512;         // TMEM columns allocated
constexpr uint32_t kColS = 0;             // S of query tile x at kColS + 64 x
constexpr uint32_t kColO = 128;           // O of query tile x at kColO + 128 x
constexpr uint32_t kColP = 384;           // P of query tile x at kColP + 32 x
constexpr int kTcWaitLimit = 1 << 22;

constexpr int kTileBytes = kTcKeys * kHeadDim * 2;           // 16 KB
constexpr int kOffQ = 0;                                      // 2 x 32 KB: Q_A, Q_B (TMA, 128-byte swizzle)
constexpr int kOffK = kOffQ + 2 * kTcQ * kHeadDim * 2;        // 3 x 16 KB: K ring (TMA, 128-byte swizzle)
constexpr int kOffVt = kOffK + kSlots * kTileBytes;           // 3 x 16 KB: V^T ring, fp16 (operand layout)
constexpr int kOffVs = kOffVt + kSlots * kTileBytes;          // 2 x 16 KB: V staging (producer, TMA, 1 KB aligned)
constexpr int kOffBar = kOffVs + 2 * kTileBytes;              // mbarriers, TMEM base, abort flag
// mbarriers: tile published, slot read by query tile A / B (per slot); S
// and P V complete, S read, P written, Q loaded (per query tile); TMA bytes
// landed (per staging tile); each issuing thread's products all complete
constexpr int kBarFull = 0, kBarEmptyA = kSlots, kBarEmptyB = 2 * kSlots, kBarS = 3 * kSlots, kBarO = kBarS + 2,
              kBarSfree = kBarO + 2, kBarPfull = kBarSfree + 2, kBarQ = kBarPfull + 2, kBarTma = kBarQ + 2,
              kBarDone = kBarTma + 2, kNumBars = kBarDone + 2;
static_assert(kOffK % 1024 == 0 && kOffVs % 1024 == 0, "the 128-byte swizzle wants 1 KB aligned boxes");
constexpr int kTcSmem = kOffBar + 8 * kNumBars + 16;

// named barriers (0 is __syncthreads)
constexpr int kNbQuery = 1;  // + query tile: 1, 2
constexpr int kNbProducer = 3;

// Staged V as TMA writes it with the 128-byte swizzle: dims [64 b, 64 b + 64)
// in box b (8 KB), row r (a key) of 128 bytes, its 16-byte chunk c at
// c ^ (r % 8), so the 8 rows an ldmatrix reads together lie on different banks.
__device__ __forceinline__ int vstage_off(int r, int c) {
  return ((c >> 3) << 13) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Byte offset of 16-byte chunk c (elements 8c .. 8c + 7) of row r in the
// operand layout of a tile with `kch` chunks per row: core matrices of 8 rows
// x 16 bytes, row groups kch * 128 bytes apart, chunks 128 bytes apart.
__device__ __forceinline__ int core_off(int r, int c, int kch) { return ((r >> 3) * kch + c) * 128 + (r & 7) * 16; }

// Shared-memory operand descriptor: K-major, no swizzle; leading byte offset
// `lbo` (between the two core matrices of a K step), stride byte offset
// `sbo` (between 8-row groups); descriptor version 1.
__device__ __forceinline__ uint64_t op_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}

// Descriptor of a K-major operand with the 128-byte swizzle (as TMA writes
// it): 8-row groups of 128-byte rows 1 KB apart; the leading byte offset is
// unused; layout type 2 at bit 61.  A K step of 16 elements advances the
// start address by 32 bytes inside the 128-byte row.
__device__ __forceinline__ uint64_t op_desc_sw128(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
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

// The same with A (M x K, K-major) read from tensor memory at `atmem`.
__device__ __forceinline__ void mma_f16_ts(uint32_t dtmem, uint32_t atmem, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(dtmem),
      "r"(atmem), "l"(b), "r"(idesc), "r"((uint32_t)acc));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void bar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(bar), "r"(bytes)
               : "memory");
}

// One TMA box of a 3-d tensor map into shared memory, counted on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void bar_arrive(uint32_t bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(bar) : "memory");
}

// Whether the mbarrier's phase `parity` has completed (does not wait).
__device__ __forceinline__ bool bar_test(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait for the mbarrier's phase `parity`; true when it completed.
// With `abort` it also gives up once another thread has set that flag.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, const volatile int* abort) {
  uint32_t done = 0;
  for (int it = 0; it < kTcWaitLimit && !done; ++it) {
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (!done && abort != nullptr && (it & 63) == 63 && *abort) break;
  }
  return done != 0;
}

// A failed wait: flag it for the host and tell the other warpgroups.
__device__ __forceinline__ void give_up(const DevState& s, volatile int* abort) {
  if (!*abort) {
    *abort = 1;
    atomicOr(&s.counters[kCtrStatus], kDevWaitTimeout);
  }
}

// Barrier over one warpgroup (named barrier `id`, 128 threads) that ANDs `v`
// across it.
__device__ __forceinline__ bool wg_and(int id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id)
      : "memory");
  return r != 0;
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

__device__ __forceinline__ void ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void st16u(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]));
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
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

// Key tiles a 128-query tile starting at q0 attends to.
__device__ __forceinline__ int key_tiles(int q0, int n) {
  return min((q0 + kTcQ - 1) / kTcKeys + 1, (n + kTcKeys - 1) / kTcKeys);
}

__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_fwd_tc_kernel(DevState s, int n, const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                          uint16_t* __restrict__ out, float* __restrict__ stats, float qk_scale_log2) {
  extern __shared__ __align__(1024) uint8_t tc_smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(tc_smem + kOffBar);
  uint32_t* tbase = reinterpret_cast<uint32_t*>(tc_smem + kOffBar + 8 * kNumBars);
  volatile int* abort = reinterpret_cast<volatile int*>(tc_smem + kOffBar + 8 * kNumBars + 4);
  auto bar = [&](int i) { return saddr(bars + i); };

  // blocks launch x fastest: a (query head, sequence)'s query blocks run
  // together, longest first, and share its K and V in L2 (ordering every
  // head's longest block first instead spread the working set past L2 and
  // was slower)
  const int qb = gridDim.x - 1 - blockIdx.x, hqi = blockIdx.y, bl = blockIdx.z;
  const int hkvi = hqi / s.group;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int role = tid / kWg, wt = tid % kWg;  // 0, 1: query tiles A, B; 2: producer; 3: MMA warp
  const size_t qrow0 = ((size_t)bl * s.hq + hqi) * n;
  const int zkv = bl * s.hkv + hkvi;  // the (sequence, KV head) plane of the K / V tensor maps
  const int qblk = qb * kTcBlock;
  const int n_a = key_tiles(qblk, n), n_kt = key_tiles(qblk + kTcQ, n);  // tile B sees the most keys

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tbase)),
                 "r"(kTcCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar(i)));
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tbase;

  if (role == 2) {
    // ---------------------------------------------------------------- producer
    __half2 vmax = __floats2half2_rn(0.0f, 0.0f);  // largest |V| in fp16 (NaN kept)
    const int pw = warp - 8;
    bool ok = true;
    int issued = 0, landed = 0;  // tiles whose copies were issued / seen complete
    // tile jt's K into its ring slot and V into staging buffer jt % 2 (one
    // thread; the staging buffer held tile jt - 2, transposed already)
    auto load = [&](int jt) {
      const uint32_t tb = bar(kBarTma + (jt & 1));
      bar_expect_tx(tb, 2 * kTileBytes);
      const uint32_t kdst = saddr(tc_smem + kOffK + (jt % kSlots) * kTileBytes);
      tma_load_3d(kdst, &tm_k, 0, jt * kTcKeys, zkv, tb);
      tma_load_3d(kdst + kTileBytes / 2, &tm_k, 64, jt * kTcKeys, zkv, tb);
      const uint32_t vdst = saddr(tc_smem + kOffVs + (jt & 1) * kTileBytes);
      tma_load_3d(vdst, &tm_v, 0, jt * kTcKeys, zkv, tb);
      tma_load_3d(vdst + kTileBytes / 2, &tm_v, 64, jt * kTcKeys, zkv, tb);
    };
    if (wt == 0) {
      // both query tiles first (128-row boxes; rows past n read as zeros)
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const uint32_t qb_bar = bar(kBarQ + x), qdst = saddr(tc_smem + kOffQ + x * (kTcQ * kHeadDim * 2));
        bar_expect_tx(qb_bar, kTcQ * kHeadDim * 2);
        tma_load_3d(qdst, &tm_q, 0, qblk + x * kTcQ, bl * s.hq + hqi, qb_bar);
        tma_load_3d(qdst + kTcQ * 128, &tm_q, 64, qblk + x * kTcQ, bl * s.hq + hqi, qb_bar);
      }
      load(0);
    }
    issued = 1;
    for (int j = 0; j < n_kt; ++j) {
      // tile j's copies complete
      if (bar_wait(bar(kBarTma + (j & 1)), (uint32_t)((j >> 1) & 1), abort)) {
        ++landed;
      } else {
        give_up(s, abort);
        ok = false;
      }
      if (!wg_and(kNbProducer, ok)) break;
      // V^T of tile j (dims x keys) in fp16: the 8 x 8 block (key group kg,
      // dim group dg) of V transposed is core matrix (dg, kg) of V^T
      const uint8_t* sv = tc_smem + kOffVs + (j & 1) * kTileBytes;
      uint8_t* svt = tc_smem + kOffVt + (j % kSlots) * kTileBytes;
#pragma unroll
      for (int bi = 0; bi < 8; ++bi) {
        const int blk = pw * 32 + bi * 4;  // 4 blocks per ldmatrix: dim groups dg .. dg + 3
        const int kg = blk >> 4, dg = blk & 15;
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
      // V^T (written) of tile j to the tensor cores' proxy; K came by TMA
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      if (!wg_and(kNbProducer, !*abort)) break;
      if (wt == 0) bar_arrive(bar(kBarFull + j % kSlots));
      // the slot of tile j + 1 held tile j + 1 - kSlots: free once tile B's
      // P V product of that tile completed (and A's, if A saw that tile)
      if (j + 1 < n_kt) {
        const int jp = j + 1 - kSlots;
        if (jp >= 0) {
          const uint32_t par = (uint32_t)((jp / kSlots) & 1);
          if (!bar_wait(bar(kBarEmptyB + jp % kSlots), par, abort) ||
              (jp < n_a && !bar_wait(bar(kBarEmptyA + jp % kSlots), par, abort))) {
            give_up(s, abort);
            ok = false;
          }
        }
        if (!wg_and(kNbProducer, ok)) break;
        if (wt == 0) load(j + 1);
        ++issued;
      }
    }
    // copies in flight (left behind after a failed wait) land before the CTA
    // goes away
    if (wt == 0)
      for (; landed < issued; ++landed) bar_wait(bar(kBarTma + (landed & 1)), (uint32_t)((landed >> 1) & 1), nullptr);
    // a saturated V entry reads 65504 in fp16, which no bf16 value converts to
    const uint32_t vmb = *reinterpret_cast<const uint32_t*>(&vmax);
    if ((vmb & 0x7FFFu) >= kF16Max || ((vmb >> 16) & 0x7FFFu) >= kF16Max)
      atomicOr(&s.counters[kCtrStatus], kDevPrefillRange);
  } else if (role == 3) {
    // ----------------------------------------------------------- MMA issuers
    const int x = warp - 12;  // the query tile this warp's thread issues for
    if (lane == 0) {
      const uint32_t id_s = instr_desc(kTcQ, kTcKeys, true);
      const uint32_t id_o = instr_desc(kTcQ, kHeadDim, false);
      const uint32_t qaddr = saddr(tc_smem + kOffQ + x * (kTcQ * kHeadDim * 2));
      const int nx = x == 0 ? n_a : n_kt;
      const int bar_empty = x == 0 ? kBarEmptyA : kBarEmptyB;
      // S(jt) = Q K(jt)^T
      auto mma_s = [&](int jt) {
        const uint32_t kaddr = saddr(tc_smem + kOffK + (jt % kSlots) * kTileBytes);
#pragma unroll
        for (int ks = 0; ks < kHeadDim / 16; ++ks)
          mma_f16(tmem + kColS + 64 * x, op_desc_sw128(qaddr + (ks >> 2) * (kTcQ * 128) + (ks & 3) * 32),
                  op_desc_sw128(kaddr + (ks >> 2) * (kTileBytes / 2) + (ks & 3) * 32), id_s, ks > 0);
        mma_commit(bar(kBarS + x));
      };
      // O += P V(jt)
      auto mma_pv = [&](int jt) {
        const uint32_t vtaddr = saddr(tc_smem + kOffVt + (jt % kSlots) * kTileBytes);
#pragma unroll
        for (int ks = 0; ks < kTcKeys / 16; ++ks)
          mma_f16_ts(tmem + kColO + 128 * x, tmem + kColP + 32 * x + 8 * ks,
                     op_desc(vtaddr + ks * 256, 128, (kTcKeys / 8) * 128), id_o, jt > 0 || ks > 0);
        mma_commit(bar(kBarO + x));
      };
      // Issue whatever is ready, in order: S(t) once tile t is published and
      // the query tile has read S(t - 1); P V(t) once it has written P(t),
      // then that slot's "empty" (only for slots the producer refills).
      // Counts of the completions seen on each barrier give the parities.
      int n_full = 0, s_next = 0, pv_next = 0, sread = 0, pwritten = 0, idle = 0;
      bool qready = false;
      while (pv_next < nx) {
        bool progress = false;
        if (n_full < nx && bar_test(bar(kBarFull + n_full % kSlots), (uint32_t)((n_full / kSlots) & 1))) {
          ++n_full;
          progress = true;
        }
        if (!qready && bar_test(bar(kBarQ + x), 0)) qready = progress = true;
        if (sread < s_next && bar_test(bar(kBarSfree + x), (uint32_t)(sread & 1))) {
          ++sread;
          progress = true;
        }
        if (pwritten < s_next && bar_test(bar(kBarPfull + x), (uint32_t)(pwritten & 1))) {
          ++pwritten;
          progress = true;
        }
        if (s_next < nx && s_next < n_full && qready && sread >= s_next) {
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          mma_s(s_next);
          ++s_next;
          progress = true;
        }
        if (pwritten > pv_next) {
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          mma_pv(pv_next);
          if (pv_next + kSlots < n_kt) mma_commit(bar(bar_empty + pv_next % kSlots));
          ++pv_next;
          progress = true;
        }
        if (progress) {
          idle = 0;
        } else if (++idle >= kTcWaitLimit || ((idle & 63) == 0 && *abort)) {
          give_up(s, abort);
          break;
        }
      }
      // every product issued here complete before the tensor memory goes back
      mma_commit(bar(kBarDone + x));
      bar_wait(bar(kBarDone + x), 0, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ query tile
    const int x = role, nb = kNbQuery + x;
    const int q0 = qblk + x * kTcQ, nx = x == 0 ? n_a : n_kt;
    const int qi = q0 + wt;  // this thread's query row
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);  // this warp's lanes
    const uint32_t col_s = kColS + 64 * x, col_o = kColO + 128 * x, col_p = kColP + 32 * x;
    const uint32_t bar_s = bar(kBarS + x), bar_o = bar(kBarO + x);
    bool ok = true;

    float m = kNegBig, l = 0.0f;
    for (int j = 0; j < nx; ++j) {
      const int k0 = j * kTcKeys;
      // S(j) complete: read this row; then S(j + 1) may overwrite it
      if (!bar_wait(bar_s, (uint32_t)(j & 1), abort)) {
        give_up(s, abort);
        ok = false;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      float xv[kTcKeys];
#pragma unroll
      for (int c0 = 0; c0 < kTcKeys; c0 += 16) ld16(trow + col_s + c0, *reinterpret_cast<float(*)[16]>(&xv[c0]));
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      if (!wg_and(nb, ok)) {
        ok = false;
        break;
      }
      if (wt == 0) bar_arrive(bar(kBarSfree + x));
      if (k0 + kTcKeys - 1 > q0 || k0 + kTcKeys > n) {
#pragma unroll
        for (int i = 0; i < kTcKeys; ++i) {
          const int ki = k0 + i;
          if (!(ki <= qi && ki < n)) xv[i] = -INFINITY;
        }
      }
      // four independent chains of maxima
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < kTcKeys; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], xv[i]);
      float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      mx *= qk_scale_log2;  // scale > 0: the maximum commutes with it
      const bool grow = mx > m + kTcLazy;
      const float alpha = grow ? fast_exp2(m - mx) : 1.0f;
      if (grow) {
        l *= alpha;
        m = mx;
      }
      // P V(j - 1) complete: O may be rescaled and P overwritten
      if (j > 0 && !bar_wait(bar_o, (uint32_t)((j - 1) & 1), abort)) {
        give_up(s, abort);
        ok = false;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      // TMEM loads and stores are warp-collective: the warp rescales when
      // any of its rows must, the others by 1
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll 1
        for (int c0 = 0; c0 < kHeadDim; c0 += 16) {
          float t[16];
          ld16(trow + col_o + c0, t);
#pragma unroll
          for (int i = 0; i < 16; ++i) t[i] *= alpha;
          st16(trow + col_o + c0, t);
        }
      }
      // P in fp16 into tensor memory, keys 2c and 2c + 1 in column c (the
      // sum adds the unrounded p, as the decode kernels do)
      const float nm = -m;
      float lp[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // four independent chains of sums
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pw[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = fast_exp2(fmaf(xv[32 * h + 2 * e], qk_scale_log2, nm));
          const float p1 = fast_exp2(fmaf(xv[32 * h + 2 * e + 1], qk_scale_log2, nm));
          lp[(2 * e) & 3] += p0;
          lp[(2 * e + 1) & 3] += p1;
          const __half2 hh = __floats2half2_rn(p0, p1);
          pw[e] = *reinterpret_cast<const uint32_t*>(&hh);
        }
        st16u(trow + col_p + 16 * h, pw);
      }
      l += (lp[0] + lp[1]) + (lp[2] + lp[3]);
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      if (!wg_and(nb, ok)) {
        ok = false;
        break;
      }
      if (wt == 0) bar_arrive(bar(kBarPfull + x));
    }
    if (ok) {
      // P V(last) complete
      if (!bar_wait(bar_o, (uint32_t)((nx - 1) & 1), abort)) {
        give_up(s, abort);
        ok = false;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      ok = wg_and(nb, ok);
    }
    if (ok) {
      // O / l to bf16, and the row's (max, sum); every lane reads (the TMEM
      // load is warp-collective), rows past n store nothing
      const bool row_ok = qi < n;
      const float inv = row_ok ? 1.0f / l : 0.0f;
      uint16_t* orow = out + (qrow0 + (row_ok ? qi : 0)) * kHeadDim;
#pragma unroll 1
      for (int c0 = 0; c0 < kHeadDim; c0 += 16) {
        float t[16];
        ld16(trow + col_o + c0, t);
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
      if (row_ok) *reinterpret_cast<float2*>(stats + (qrow0 + qi) * 2) = make_float2(m, l);
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcCols));
}

// ---------------------------------------------------------------------------
// Prompt H2O scores on the tensor cores: every prompt key's score is the sum,
// over the later queries of the query heads of its KV head, of its
// probability exp2(s log2e / sqrt(d) - m_q) / l_q, with the forward kernel's
// row statistics (m_q, l_q).
//
// One 320-thread CTA per (128-key tile, KV head, sequence), two per SM, keys
// on the TMEM lanes: S^T (128 keys x 128 queries) = K Q^T by tcgen05.mma (M
// 128, N 128, bf16: exact products; K from shared memory once, by TMA, with
// the 128-byte swizzle; the query tile by TMA into a ring of two slots), so
// thread t of a warpgroup owns key t's row and adds its probabilities in a
// register.  Roles: warpgroups 0 and 1 take alternate query blocks (TMEM
// columns [0, 128) and [128, 256)); warp 8 loads the query tiles and stages
// b_q = m_q + log2(l_q) per query (+inf past the prompt, so those read as
// zero); warp 9 issues the products from one thread.  Query blocks are (query
// head g of the group, 128-query tile qt >= the key tile); only the diagonal
// block needs the causal mask.  The two warpgroups' sums meet in shared
// memory and go straight into the sink, pool or window score slot of each
// key (one CTA owns a key tile, so no atomics).
constexpr int kScThreads = 2 * kWg + 64;
constexpr int kScTile = 128;                                  // keys per CTA, queries per block
constexpr int kScTileBytes = kScTile * kHeadDim * 2;          // 32 KB
constexpr int kScOffK = 0;                                    // 32 KB: K (TMA, 128-byte swizzle)
constexpr int kScOffQ = kScOffK + kScTileBytes;               // 2 x 32 KB: query tiles
constexpr int kScOffB = kScOffQ + 2 * kScTileBytes;           // 2 x 512 B: b_q per slot
constexpr int kScOffRed = kScOffB + 2 * kScTile * 4;          // 512 B: warpgroup 0's sums
constexpr int kScOffBar = kScOffRed + kScTile * 4;
constexpr int kScBarK = 0, kScBarFull = 1, kScBarEmpty = 3, kScBarS = 5, kScBarSfree = 7, kScBarDone = 9,
              kScNumBars = 10;
constexpr int kScSmem = kScOffBar + 8 * kScNumBars + 16;
constexpr uint32_t kScCols = 256;

__global__ void __launch_bounds__(kScThreads, 2)
    prefill_scores_tc_kernel(DevState s, int n, const __grid_constant__ CUtensorMap tm_q,
                             const __grid_constant__ CUtensorMap tm_k, const float* __restrict__ stats,
                             float qk_scale_log2, int seq_begin) {
  extern __shared__ __align__(1024) uint8_t sc_smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(sc_smem + kScOffBar);
  uint32_t* tbase = reinterpret_cast<uint32_t*>(sc_smem + kScOffBar + 8 * kScNumBars);
  volatile int* abort = reinterpret_cast<volatile int*>(sc_smem + kScOffBar + 8 * kScNumBars + 4);
  auto bar = [&](int i) { return saddr(bars + i); };

  const int kt = blockIdx.x, h = blockIdx.y, bl = blockIdx.z;  // key tile 0 sees the most queries
  const int b = seq_begin + bl, G = s.group;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k0 = kt * kScTile;
  const int n_qt = (n + kScTile - 1) / kScTile;
  const int per_head = n_qt - kt, iters = G * per_head;  // blocks (g, qt >= kt)

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tbase)),
                 "r"(kScCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int i = 0; i < kScNumBars; ++i) {
      const uint32_t cnt = (i == kScBarFull || i == kScBarFull + 1 || i == kScBarEmpty || i == kScBarEmpty + 1) ? 2 : 1;
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar(i)), "r"(cnt));
    }
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tbase;
  float score = 0.0f;  // this thread's key, over this warpgroup's blocks

  if (warp == 8) {
    // ------------------------------------------------- query tiles and b_q
    float* sb = reinterpret_cast<float*>(sc_smem + kScOffB);
    if (lane == 0) {
      bar_expect_tx(bar(kScBarK), kScTileBytes);
      const uint32_t kdst = saddr(sc_smem + kScOffK);
      tma_load_3d(kdst, &tm_k, 0, k0, bl * s.hkv + h, bar(kScBarK));
      tma_load_3d(kdst + kScTileBytes / 2, &tm_k, 64, k0, bl * s.hkv + h, bar(kScBarK));
    }
    for (int it = 0; it < iters; ++it) {
      const int x = it & 1, g = it / per_head, qt = kt + it % per_head;
      bool ok = true;
      // the slot's previous block read (its product complete, b_q used)
      if (lane == 0 && it >= 2 && !bar_wait(bar(kScBarEmpty + x), (uint32_t)(((it - 2) >> 1) & 1), abort)) {
        give_up(s, abort);
        ok = false;
      }
      if (!__all_sync(0xffffffffu, ok)) break;
      if (lane == 0) {
        bar_expect_tx(bar(kScBarFull + x), kScTileBytes);
        const uint32_t qdst = saddr(sc_smem + kScOffQ + x * kScTileBytes);
        const int plane = bl * s.hq + h * G + g;
        tma_load_3d(qdst, &tm_q, 0, qt * kScTile, plane, bar(kScBarFull + x));
        tma_load_3d(qdst + kScTileBytes / 2, &tm_q, 64, qt * kScTile, plane, bar(kScBarFull + x));
      }
      const size_t srow = ((size_t)bl * s.hq + h * G + g) * n + (size_t)qt * kScTile;
#pragma unroll
      for (int e = 0; e < kScTile / 32; ++e) {
        const int i = lane + 32 * e;
        float bq = INFINITY;
        if (qt * kScTile + i < n) {
          const float2 st = *reinterpret_cast<const float2*>(stats + (srow + i) * 2);
          bq = st.x + log2f(st.y);
        }
        sb[x * kScTile + i] = bq;
      }
      __syncwarp();
      if (lane == 0) bar_arrive(bar(kScBarFull + x));
    }
  } else if (warp == 9) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_s = instr_desc(kScTile, kScTile, true);
      const uint32_t kaddr = saddr(sc_smem + kScOffK);
      bool ok = bar_wait(bar(kScBarK), 0, abort);
      if (!ok) give_up(s, abort);
      for (int it = 0; ok && it < iters; ++it) {
        const int x = it & 1;
        if (!bar_wait(bar(kScBarFull + x), (uint32_t)((it >> 1) & 1), abort) ||
            (it >= 2 && !bar_wait(bar(kScBarSfree + x), (uint32_t)(((it - 2) >> 1) & 1), abort))) {
          give_up(s, abort);
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t qaddr = saddr(sc_smem + kScOffQ + x * kScTileBytes);
#pragma unroll
        for (int ks = 0; ks < kHeadDim / 16; ++ks) {
          const uint32_t off = (ks >> 2) * (kScTileBytes / 2) + (ks & 3) * 32;
          mma_f16(tmem + 128 * x, op_desc_sw128(kaddr + off), op_desc_sw128(qaddr + off), id_s, ks > 0);
        }
        mma_commit(bar(kScBarS + x));
        mma_commit(bar(kScBarEmpty + x));
      }
      // every product issued here complete before the tensor memory goes back
      mma_commit(bar(kScBarDone));
      bar_wait(bar(kScBarDone), 0, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ sums over the queries
    const int x = tid / kWg, t = tid % kWg;  // warpgroup x takes blocks x, x + 2, ...
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16) + 128 * x;
    const float* sb = reinterpret_cast<const float*>(sc_smem + kScOffB) + x * kScTile;
    bool ok = true;
    for (int it = x; it < iters; it += 2) {
      const int qt = kt + it % per_head;
      if (!bar_wait(bar(kScBarS + x), (uint32_t)((it >> 1) & 1), abort) ||
          !bar_wait(bar(kScBarFull + x), (uint32_t)((it >> 1) & 1), abort)) {
        give_up(s, abort);
        ok = false;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      // four partial sums (independent add chains); queries below this key
      // only on the diagonal block, which alone takes the masked loop
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (qt != kt) {
#pragma unroll 1
        for (int c0 = 0; c0 < kScTile; c0 += 32) {
          float v[32];
          ld32(trow + c0, v);
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 b4 = *reinterpret_cast<const float4*>(sb + c0 + i);
            acc[0] += fast_exp2(fmaf(v[i], qk_scale_log2, -b4.x));
            acc[1] += fast_exp2(fmaf(v[i + 1], qk_scale_log2, -b4.y));
            acc[2] += fast_exp2(fmaf(v[i + 2], qk_scale_log2, -b4.z));
            acc[3] += fast_exp2(fmaf(v[i + 3], qk_scale_log2, -b4.w));
          }
        }
      } else {
#pragma unroll 1
        for (int c0 = 0; c0 < kScTile; c0 += 32) {
          float v[32];
          ld32(trow + c0, v);
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 b4 = *reinterpret_cast<const float4*>(sb + c0 + i);
            const float bb[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float p = fast_exp2(fmaf(v[i + e], qk_scale_log2, -bb[e]));
              acc[e] += c0 + i + e < t ? 0.0f : p;
            }
          }
        }
      }
      score += (acc[0] + acc[1]) + (acc[2] + acc[3]);
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      if (!wg_and(kNbQuery + x, ok)) break;
      if (t == 0) {
        bar_arrive(bar(kScBarSfree + x));
        bar_arrive(bar(kScBarEmpty + x));
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  // warpgroup 0's sums meet warpgroup 1's; warpgroup 1 writes the scores
  float* red = reinterpret_cast<float*>(sc_smem + kScOffRed);
  if (tid < kWg) red[tid] = score;
  __syncthreads();
  if (tid >= kWg && tid < 2 * kWg && !*abort) {
    const int t = tid - kWg, p = k0 + t;
    if (p < n) {
      const float v = score + red[t];
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
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kScCols));
}

}  // namespace

int prefill_fwd_tc_smem_bytes() { return kTcSmem; }

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn tensor_map_encoder() {
  static const EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) !=
            cudaSuccess ||
        qr != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// A [planes][n][128] bf16 tensor as a 3-d tensor map with 64 x `rows` x 1
// boxes (64 dims) and the 128-byte swizzle; rows past n read as zeros.
bool encode_kv_map(CUtensorMap* map, const uint16_t* base, int n, int planes, int rows) {
  const EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)n, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)n * kHeadDim * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_prefill_scores_tc(const DevState& s, int seq_begin, int batch, int n, const uint16_t* q,
                                    const uint16_t* k, const float* stats, float qk_scale_log2, cudaStream_t st) {
  static int done[64] = {0};
  const cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(prefill_scores_tc_kernel), kScSmem, done);
  if (e != cudaSuccess) return e;
  CUtensorMap tm_q, tm_k;
  if (!encode_kv_map(&tm_q, q, n, batch * s.hq, kScTile) || !encode_kv_map(&tm_k, k, n, batch * s.hkv, kScTile))
    return cudaErrorInvalidValue;
  const int tiles = (n + kScTile - 1) / kScTile;
  prefill_scores_tc_kernel<<<dim3(tiles, s.hkv, batch), kScThreads, kScSmem, st>>>(s, n, tm_q, tm_k, stats,
                                                                                    qk_scale_log2, seq_begin);
  return cudaGetLastError();
}

cudaError_t launch_prefill_fwd_tc(const DevState& s, int batch, int n, const uint16_t* q, const uint16_t* k,
                                  const uint16_t* v, uint16_t* out, float* stats, float qk_scale_log2,
                                  cudaStream_t st) {
  static int done[64] = {0};
  const cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(prefill_fwd_tc_kernel), kTcSmem, done);
  if (e != cudaSuccess) return e;
  CUtensorMap tm_q, tm_k, tm_v;
  if (!encode_kv_map(&tm_q, q, n, batch * s.hq, kTcQ) || !encode_kv_map(&tm_k, k, n, batch * s.hkv, kTcKeys) ||
      !encode_kv_map(&tm_v, v, n, batch * s.hkv, kTcKeys))
    return cudaErrorInvalidValue;
  const int blocks = (n + kTcBlock - 1) / kTcBlock;
  prefill_fwd_tc_kernel<<<dim3(blocks, s.hq, batch), kTcThreads, kTcSmem, st>>>(s, n, tm_q, tm_k, tm_v, out, stats,
                                                                                qk_scale_log2);
  return cudaGetLastError();
}

}  // namespace kvc
