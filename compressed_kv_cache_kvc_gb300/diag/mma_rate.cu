// Issue-rate microbenchmark of tcgen05.mma kind::f16 on this GPU: one CTA per
// SM (152), 2048 products per CTA into tensor memory from shared-memory
// operands of zeros, issued by 1, 2 or 4 warps (one thread each); prints the
// cycles per product one issuing warp sees and the TFLOP/s over the GPU.
// Every wait is bounded.  Build and run:
//   nvcc -gencode arch=compute_103a,code=sm_103a -O2 -o mma_rate mma_rate.cu && ./mma_rate
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
__device__ __forceinline__ uint32_t sa(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t desc_ns(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}
__global__ void __launch_bounds__(128, 1) rate(int mode, int reps, unsigned long long* out, int* flag, int issuers) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ __align__(8) uint64_t mbars[4];
  __shared__ uint32_t tb;
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < 64 * 1024 / 16; i += 128) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(sa(&tb)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int b = 0; b < 4; ++b) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sa(&mbars[b])));
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  asm volatile("fence.proxy.async.shared::cta;");
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tmem = tb;
  if ((tid & 31) == 0 && warp < issuers) {
    const uint64_t& mbar = mbars[warp];
    // modes: 0 M128 N64 (ss), 1 M128 N128 (ss), 2 M128 N256 (ss), 3 M128 N128 (A in TMEM), 4 M128 N64 ss, 4 accumulators round robin
    const int N = mode == 0 || mode == 4 ? 64 : (mode == 2 ? 256 : 128);
    const uint32_t id = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    const uint32_t idh = (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    const uint64_t da = desc_ns(sa(sm), 128, 2048), db = desc_ns(sa(sm + 32768), 128, 256);  // B: 32 row groups x 256 B stay inside the 32 KB half
    const long long t0 = clock64();
    for (int r = 0; r < reps / issuers; ++r) {
      const uint32_t d = mode == 4 ? tmem + 64 * (r & 3) : tmem + (issuers > 1 ? 128 * warp : 0);
      if (mode == 3)
        asm volatile("{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
                     ::"r"(tmem + 256), "r"(tmem), "l"(db), "r"(idh), "r"(1u));
      else
        asm volatile("{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                     ::"r"(d), "l"(da), "l"(db), "r"(id), "r"(1u));
    }
    const long long t1 = clock64();
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(sa(&mbar)));
    uint32_t done = 0;
    for (int it = 0; it < (1 << 24) && !done; ++it)
      asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
                   : "=r"(done) : "r"(sa(&mbar)), "r"(0));
    const long long t2 = clock64();
    if (!done) atomicOr(flag, 1);
    if (blockIdx.x == 0 && warp == 0) { out[0] = t1 - t0; out[1] = t2 - t0; }
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
}
int main() {
  unsigned long long* d; int* f; cudaMalloc(&d, 16); cudaMalloc(&f, 4); cudaMemset(f, 0, 4);
  cudaFuncSetAttribute(rate, cudaFuncAttributeMaxDynamicSharedMemorySize, 65536);
  const char* names[5] = {"M128 N64 K16 ss", "M128 N128 K16 ss", "M128 N256 K16 ss", "M128 N128 K16 ts(A tmem)", "M128 N64 ss, 4 accumulators"};
  const double flop[5] = {128.0 * 64 * 16 * 2, 128.0 * 128 * 16 * 2, 128.0 * 256 * 16 * 2, 128.0 * 128 * 16 * 2, 128.0 * 64 * 16 * 2};
  for (int cfg = 0; cfg < 9; ++cfg) {
    const int mode = cfg < 5 ? cfg : (cfg < 7 ? 0 : 1), issuers = cfg < 5 ? 1 : (cfg == 5 || cfg == 7 ? 2 : 4);
    const int reps = 2048;
    rate<<<152, 128, 65536>>>(mode, reps, d, f, issuers);
    cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
    cudaEventRecord(e0);
    rate<<<152, 128, 65536>>>(mode, reps, d, f, issuers);
    cudaEventRecord(e1);
    cudaError_t e = cudaDeviceSynchronize();
    float ms; cudaEventElapsedTime(&ms, e0, e1);
    unsigned long long h[2]; int hf; cudaMemcpy(h, d, 16, cudaMemcpyDeviceToHost); cudaMemcpy(&hf, f, 4, cudaMemcpyDeviceToHost);
    printf("issuers %d  %-30s err=%s flag=%d issue %.1f cyc/mma, complete %.1f cyc/mma, %.0f TFLOP/s (152 SMs)\n", issuers, names[mode], cudaGetErrorString(e), hf,
           (double)h[0] / reps, (double)h[1] / reps, flop[mode] * reps * 152 / (ms * 1e-3) / 1e12);
    if (e != cudaSuccess) return 1;
  }
  return 0;
}
