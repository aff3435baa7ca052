// pipe_rate.cu -- issue rate of the instruction classes an in-register weight
// dequantiser is built from, on one SM: each thread runs 8 independent
// dependency chains of one instruction, so the rate is the pipe's throughput,
// not its latency.  Build and run:
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o pipe_rate pipe_rate.cu && ./pipe_rate
#include <cstdint>
#include <cstdio>
#include <cuda_runtime.h>

constexpr int kChains = 8;

template <int OP>
__global__ void __launch_bounds__(1024) pipe_kernel(uint32_t* out, long long* cycles, int iters, uint32_t seed) {
  uint32_t v[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c) v[c] = seed * (threadIdx.x + 1) + c * 0x9E3779B9u;
  const uint32_t m = 0x000F000Fu ^ seed, k = 0x43084308u + seed, sh = 3u + (seed & 1u);
  __syncthreads();
  const long long t0 = clock64();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) {
      if (OP == 0) asm volatile("lop3.b32 %0, %0, %1, %2, 0x6A;" : "+r"(v[c]) : "r"(m), "r"(k));
      if (OP == 1) asm volatile("prmt.b32 %0, %0, %1, 0x5140;" : "+r"(v[c]) : "r"(k));
      if (OP == 2) asm volatile("shf.r.clamp.b32 %0, %0, %1, %2;" : "+r"(v[c]) : "r"(k), "r"(sh));
      if (OP == 3) asm volatile("mul.hi.u32 %0, %0, %1;" : "+r"(v[c]) : "r"(k));
      if (OP == 4) asm volatile("mad.lo.u32 %0, %0, %1, %2;" : "+r"(v[c]) : "r"(k), "r"(m));
      if (OP == 5) asm volatile("add.u32 %0, %0, %1;" : "+r"(v[c]) : "r"(k));
      if (OP == 6) asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+r"(v[c]) : "r"(k), "r"(m));
      if (OP == 7) asm volatile("fma.rn.bf16x2 %0, %0, %1, %2;" : "+r"(v[c]) : "r"(k), "r"(m));
      if (OP == 8) asm volatile("sub.rn.bf16x2 %0, %0, %1;" : "+r"(v[c]) : "r"(k));
    }
  }
  __syncthreads();
  const long long t1 = clock64();
  uint32_t acc = 0;
#pragma unroll
  for (int c = 0; c < kChains; ++c) acc ^= v[c];
  out[blockIdx.x * blockDim.x + threadIdx.x] = acc;
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

template <int OP>
void run(const char* name, uint32_t* out, long long* cycles, int threads) {
  const int iters = 4096;
  pipe_kernel<OP><<<1, threads>>>(out, cycles, iters, 7);
  pipe_kernel<OP><<<1, threads>>>(out, cycles, iters, 7);
  long long c = 0;
  cudaMemcpy(&c, cycles, 8, cudaMemcpyDeviceToHost);
  const double ops = double(iters) * kChains * threads;
  printf("  %-12s %4d threads: %6.1f lane-ops/clk/SM = %.2f warp-instructions/clk per scheduler\n", name, threads,
         ops / c, ops / c / 32 / 4);
}

int main() {
  uint32_t* out;
  long long* cycles;
  if (cudaMalloc(&out, 1024 * 4) != cudaSuccess || cudaMalloc(&cycles, 8) != cudaSuccess) return 1;
  for (int th : {256, 1024}) {
    run<0>("lop3", out, cycles, th);
    run<1>("prmt", out, cycles, th);
    run<2>("shf.r", out, cycles, th);
    run<3>("mul.hi.u32", out, cycles, th);
    run<4>("mad.lo.u32", out, cycles, th);
    run<5>("add.u32", out, cycles, th);
    run<6>("fma.f32", out, cycles, th);
    run<7>("fma.bf16x2", out, cycles, th);
    run<8>("sub.bf16x2", out, cycles, th);
  }
  const cudaError_t e = cudaDeviceSynchronize();
  printf("%s\n", cudaGetErrorString(e));
  return e == cudaSuccess ? 0 : 1;
}
