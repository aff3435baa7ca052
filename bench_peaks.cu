// bench_peaks.cu -- dense tensor-core peaks of this GPU for the MMA kinds the
// MoE layer's GEMMs issue, measured with tcgen05 instructions (bench.py --peaks).
//
// Every SM runs one CTA whose single issuing thread sends `iters` MMAs
// (M = 128) back to back, round-robin over `nacc` TMEM accumulators, then
// waits once (bounded) for them to retire.  Operands sit in shared memory in
// the 128-byte-swizzle K-major layout; their values do not change the rate.
// FLOPs = 2 * M * N * K per MMA; time = CUDA events around the launch.
//   kind::f16            BF16 x BF16 -> FP32, K = 16 per instruction
//   kind::mxf4nvf4       E2M1 x E2M1 with UE4M3 scales per 16 -> FP32, K = 64
// Prints one JSON line: the best rate of each kind over the N / accumulator
// shapes tried, and every shape's rate.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <vector>

namespace {

__device__ __forceinline__ uint32_t sh_addr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Smem operand descriptor: K-major, 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t operand_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (64ull << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptors (M = 128, both operands K-major, FP32 accumulation).
__host__ __device__ constexpr uint32_t desc_bf16(int n) { return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | (8u << 24); }
__host__ __device__ constexpr uint32_t desc_nvf4(int n) { return (1u << 7) | (1u << 10) | ((n >> 3) << 17) | (8u << 24); }

constexpr uint64_t kLimitNs = 2000000000ull;

__global__ void __launch_bounds__(128, 1) peak_kernel(int fp4, int n, int nacc, int iters, int* status) {
  extern __shared__ uint8_t dyn[];
  uint8_t* a_tile = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* b_tile = a_tile + 128 * 128;
  __shared__ uint64_t done;
  __shared__ uint32_t tmem_base;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sh_addr(&done)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(sh_addr(&tmem_base)) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // operands: E2M1 1.0 pairs (0x22) for FP4, BF16 zeros otherwise
  for (int i = threadIdx.x; i < 128 * 128 + 256 * 128; i += blockDim.x) a_tile[i] = fp4 ? 0x22 : 0;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_base;
  const uint32_t sf_col = static_cast<uint32_t>(nacc * n);  // scale factors after the accumulators
  if (fp4) {
    // UE4M3 1.0 in every byte of 16 columns, every lane (each warp its lane quarter)
    const uint32_t one = 0x38383838u;
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1};" ::"r"(
            tmem + (static_cast<uint32_t>(warp * 32) << 16) + sf_col),
        "r"(one)
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (threadIdx.x == 0) {
    const uint64_t ad = operand_desc(sh_addr(a_tile)), bd = operand_desc(sh_addr(b_tile));
    const uint32_t id = fp4 ? desc_nvf4(n) : desc_bf16(n);
    int acc = 0;
    for (int i = 0; i < iters; ++i) {
      const uint32_t d = tmem + static_cast<uint32_t>(acc * n);
      const uint64_t kstep = static_cast<uint64_t>((i >> 2) & 3) * 2;  // 32-byte steps inside the row
      const uint32_t accumulate = i >= nacc;
      if (fp4) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
            "l"(ad + kstep), "l"(bd + kstep), "r"(id), "r"(tmem + sf_col), "r"(tmem + sf_col + 8), "r"(accumulate)
            : "memory");
      } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
            "l"(ad + kstep), "l"(bd + kstep), "r"(id), "r"(accumulate)
            : "memory");
      }
      if (++acc == nacc) acc = 0;
    }
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(sh_addr(&done)) : "memory");
    const uint64_t t0 = now_ns();
    uint32_t ok = 0;
    while (!ok) {
      asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                   : "=r"(ok)
                   : "r"(sh_addr(&done))
                   : "memory");
      if (!ok && now_ns() - t0 > kLimitNs) {
        atomicOr(status, 1);
        break;
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

struct Shape {
  int fp4, n, nacc;
};

}  // namespace

int main() {
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0) != cudaSuccess) return 1;
  const int smem = 128 * 128 + 256 * 128 + 1024;
  if (cudaFuncSetAttribute(peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 1;
  int* status = nullptr;
  if (cudaMalloc(&status, sizeof(int)) != cudaSuccess || cudaMemset(status, 0, sizeof(int)) != cudaSuccess) return 1;
  const Shape shapes[] = {{0, 256, 1}, {0, 128, 2}, {0, 128, 3}, {1, 256, 1}, {1, 128, 2}, {1, 128, 3}, {1, 64, 4}};
  const int iters = 16384;
  double best[2] = {0, 0};
  std::vector<double> rates;
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  for (const Shape& s : shapes) {
    peak_kernel<<<sms, 128, smem>>>(s.fp4, s.n, s.nacc, 512, status);  // warm-up
    double best_here = 0;
    for (int rep = 0; rep < 3; ++rep) {
      cudaEventRecord(e0);
      peak_kernel<<<sms, 128, smem>>>(s.fp4, s.n, s.nacc, iters, status);
      cudaEventRecord(e1);
      if (cudaEventSynchronize(e1) != cudaSuccess) return 1;
      float ms = 0;
      cudaEventElapsedTime(&ms, e0, e1);
      const double k = s.fp4 ? 64.0 : 16.0;
      const double tflops = 2.0 * 128 * s.n * k * iters * sms / (ms * 1e-3) / 1e12;
      if (tflops > best_here) best_here = tflops;
    }
    rates.push_back(best_here);
    if (best_here > best[s.fp4]) best[s.fp4] = best_here;
  }
  int st = 0;
  cudaMemcpy(&st, status, sizeof(int), cudaMemcpyDeviceToHost);
  if (st || cudaGetLastError() != cudaSuccess) {
    printf("{\"error\": \"a wait ran out or a launch failed\"}\n");
    return 1;
  }
  printf("{\"f16_tflops\": %.1f, \"mxf4nvf4_tflops\": %.1f, \"sms\": %d, \"iters_per_cta\": %d, \"shapes\": [", best[0],
         best[1], sms, iters);
  for (size_t i = 0; i < rates.size(); ++i)
    printf("%s{\"kind\": \"%s\", \"n\": %d, \"acc\": %d, \"tflops\": %.1f}", i ? ", " : "",
           shapes[i].fp4 ? "mxf4nvf4" : "f16", shapes[i].n, shapes[i].nacc, rates[i]);
  printf("]}\n");
  return 0;
}
