// mma_rate.cu -- how many SM cycles one tensor-core instruction costs on this GPU:
// tcgen05.mma kind::f16 (M = 128, N = 16..256, A from shared or tensor memory)
// against the warp-level mma.sync m16n8k16 BF16.  Operands are zeros; one CTA
// per SM; the only wait is bounded.  Build and run:
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -o mma_rate mma_rate.cu && ./mma_rate
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
#include "../csrc/mnw_ptx.cuh"
using namespace mnw;

__global__ void __launch_bounds__(128, 1) tc_rate(int N, int ts, int iters, unsigned long long* out, unsigned* err) {
  extern __shared__ __align__(1024) uint8_t sm[];
  uint8_t* s = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  for (int i = threadIdx.x; i < (48 << 10) / 16; i += blockDim.x) reinterpret_cast<uint4*>(s)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) { mbar_init(&bar, 1); fence_barrier_init(); }
  if (threadIdx.x < 32) { tmem_alloc(&tbase, 512); tmem_relinquish(); }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = tbase;
  if (threadIdx.x == 0) {
    const uint32_t idesc = idesc_f16(128, N, true);
    const uint32_t a_s = smem_u32(s), b_s = smem_u32(s + 16384);
    unsigned long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
      const int kk = i & 3;
      const uint64_t bd = sdesc_sw128(b_s + kk * 32);
      if (ts) mma_ts(tm + 256, tm + kk * 8, bd, idesc, i > 0);
      else mma_ss(tm + 256, sdesc_sw128(a_s + kk * 32), bd, idesc, i > 0);
    }
    unsigned long long t1 = clock64();
    mma_commit(&bar);
    const uint64_t g0 = globaltimer();
    while (!mbar_try_wait(&bar, 0)) { if (globaltimer() - g0 > 1000000000ull) { atomicOr(err, 1u); break; } }
    unsigned long long t2 = clock64();
    if (blockIdx.x == 0) { out[0] = t1 - t0; out[1] = t2 - t0; }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) { tc_fence_after(); tmem_dealloc(tm, 512); }
}

// Cost of tcgen05.commit in the issuing thread: TS MMAs (M = 128, N = 64,
// A from TMEM) alternating two accumulators like a gate/up pair, a commit to
// an mbarrier after every C MMAs (C = 0: none); with WAIT the thread then
// waits for that commit's phase (each barrier's own parity), as a producer
// of a ring would.  Cadence and mode are compile-time, so the loop holds
// nothing but the MMAs, the descriptors and the commits.
template <int C, bool WAIT>
__global__ void __launch_bounds__(128, 1) tc_commit_rate(int iters, unsigned long long* out, unsigned* err) {
  extern __shared__ __align__(1024) uint8_t sm[];
  uint8_t* s = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bars[5];
  __shared__ uint32_t tbase;
  for (int i = threadIdx.x; i < (48 << 10) / 16; i += blockDim.x) reinterpret_cast<uint4*>(s)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
  }
  if (threadIdx.x < 32) { tmem_alloc(&tbase, 512); tmem_relinquish(); }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = tbase;
  if (threadIdx.x == 0) {
    const uint32_t idesc = idesc_f16(128, 64, true);
    const uint32_t b_s = smem_u32(s + 16384);
    uint32_t phase = 0;  // bit b: parity of barrier b's next phase
    unsigned long long t0 = clock64();
    for (int i = 0; i < iters; i += 8) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int kk = (u >> 1) & 3, m = u & 1;
        mma_ts(tm + 256 + m * 64, tm + kk * 8 + m * 32, sdesc_sw128(b_s + kk * 32), idesc, (i | u) > 1);
        if (C > 0 && C <= 8 && ((u + 1) % C) == 0) {
          const int b = ((i + u) / C) & 3;
          mma_commit(&bars[b]);
          if (WAIT) {
            const uint64_t g0 = globaltimer();
            while (!mbar_try_wait(&bars[b], (phase >> b) & 1)) {
              if (globaltimer() - g0 > 1000000000ull) { atomicOr(err, 2u); break; }
            }
            phase ^= 1u << b;
          }
        }
      }
      if (C > 8 && ((i + 8) % C) == 0) mma_commit(&bars[(i / C) & 3]);
    }
    unsigned long long t1 = clock64();
    mma_commit(&bars[4]);
    const uint64_t g0 = globaltimer();
    while (!mbar_try_wait(&bars[4], 0)) { if (globaltimer() - g0 > 1000000000ull) { atomicOr(err, 1u); break; } }
    unsigned long long t2 = clock64();
    if (blockIdx.x == 0) { out[0] = t1 - t0; out[1] = t2 - t0; }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) { tc_fence_after(); tmem_dealloc(tm, 512); }
}

template <int C, bool WAIT>
void commit_case(int sms, int iters, unsigned long long* d_out, unsigned* d_err, const char* what) {
  cudaFuncSetAttribute(tc_commit_rate<C, WAIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 << 10);
  cudaMemset(d_err, 0, 4);
  for (int rep = 0; rep < 2; ++rep) tc_commit_rate<C, WAIT><<<sms, 128, 64 << 10>>>(iters, d_out, d_err);
  cudaError_t e = cudaDeviceSynchronize();
  unsigned long long h[2]; cudaMemcpy(h, d_out, 16, cudaMemcpyDeviceToHost);
  unsigned herr; cudaMemcpy(&herr, d_err, 4, cudaMemcpyDeviceToHost);
  printf("tcgen05 TS N=64, 2 accumulators, %-28s issue %6.1f cyc/mma, complete %6.1f cyc/mma err=%u %s\n", what,
         h[0] / double(iters), h[1] / double(iters), herr, cudaGetErrorString(e));
}

// mma.sync m16n8k16 bf16 throughput: each warp runs 4 independent accumulator chains.
__global__ void __launch_bounds__(256) hmma_rate(int iters, unsigned long long* out, float* sink) {
  uint32_t a0 = threadIdx.x, a1 = a0 * 3, a2 = a0 * 5, a3 = a0 * 7, b0 = a0 * 11, b1 = a0 * 13;
  float c[4][4] = {};
  __syncthreads();
  unsigned long long t0 = clock64();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                   : "+f"(c[j][0]), "+f"(c[j][1]), "+f"(c[j][2]), "+f"(c[j][3])
                   : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  __syncthreads();
  unsigned long long t1 = clock64();
  if (blockIdx.x == 0 && threadIdx.x == 0) out[2] = t1 - t0;
  float acc = 0; for (int j = 0; j < 4; ++j) for (int q = 0; q < 4; ++q) acc += c[j][q];
  if (acc == 12345.f) sink[0] = acc;
}

int main() {
  int sms; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  unsigned long long* d_out; unsigned* d_err; float* d_sink;
  cudaMalloc(&d_out, 64); cudaMalloc(&d_err, 4); cudaMalloc(&d_sink, 4); cudaMemset(d_err, 0, 4);
  cudaFuncSetAttribute(tc_rate, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 << 10);
  const int iters = 4096;
  for (int ts = 0; ts < 2; ++ts)
    for (int N : {16, 32, 64, 128, 256}) {
      for (int rep = 0; rep < 2; ++rep) tc_rate<<<sms, 128, 64 << 10>>>(N, ts, iters, d_out, d_err);
      cudaError_t e = cudaDeviceSynchronize();
      unsigned long long h[2]; cudaMemcpy(h, d_out, 16, cudaMemcpyDeviceToHost);
      unsigned herr; cudaMemcpy(&herr, d_err, 4, cudaMemcpyDeviceToHost);
      printf("tcgen05 %s M=128 N=%3d: issue %.1f cyc/mma, complete %.1f cyc/mma  (%.0f MAC/clk) err=%u %s\n",
             ts ? "TS" : "SS", N, h[0] / double(iters), h[1] / double(iters),
             128.0 * N * 16 * iters / h[1], herr, cudaGetErrorString(e));
    }
  commit_case<0, false>(sms, iters, d_out, d_err, "no commit:");
  commit_case<16, false>(sms, iters, d_out, d_err, "commit every 16:");
  commit_case<8, false>(sms, iters, d_out, d_err, "commit every 8:");
  commit_case<4, false>(sms, iters, d_out, d_err, "commit every 4:");
  commit_case<2, false>(sms, iters, d_out, d_err, "commit every 2:");
  commit_case<8, true>(sms, iters, d_out, d_err, "commit every 8 and wait:");
  commit_case<4, true>(sms, iters, d_out, d_err, "commit every 4 and wait:");
  for (int warps : {4, 8, 16}) {
    hmma_rate<<<sms, warps * 32>>>(2048, d_out, d_sink);
    cudaDeviceSynchronize();
    unsigned long long h[3]; cudaMemcpy(h, d_out, 24, cudaMemcpyDeviceToHost);
    const double n_hmma = 2048.0 * 4 * warps;
    printf("mma.sync m16n8k16 bf16, %2d warps/SM: %.2f cyc per HMMA per SM (%.0f MAC/clk)\n", warps, h[2] / n_hmma,
           n_hmma * 2048 / h[2]);
  }
  return 0;
}
