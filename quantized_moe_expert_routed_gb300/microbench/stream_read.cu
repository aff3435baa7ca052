// stream_read.cu -- how fast a kernel can read a weight-sized tensor from HBM
// on this GPU, and what the L2 flush between timed runs does to the number.
//
//   part A: plain 16-byte loads over the first S bytes of a 2 GiB buffer,
//           timed after (1) writing a 512 MiB buffer (leaves dirty lines in
//           L2) or (2) writing it and then reading another 512 MiB buffer
//           (the write-back happens before the timed kernel).
//   part B: a persistent kernel pulling a [256][1024 rows][1024 B] tensor
//           (256 MiB, shaped like one expert matrix per slice) through a
//           shared-memory ring: one thread issues 2D/3D TMA boxes of W bytes
//           x 128 rows, two boxes per stage, S stages; 8 warps only wait and
//           release.  Clean L2 before each run.
//
// Every wait is bounded (mnw_ptx.cuh).  Build and run:
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -o stream_read stream_read.cu -lcuda && ./stream_read
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdio>

#include "../csrc/mnw_ptx.cuh"
using namespace mnw;

constexpr int kMaxS = 16;
struct RingBars {
  uint64_t full[kMaxS], empty[kMaxS];
  int abort;
};

__global__ void __launch_bounds__(512) read_kernel(const uint4* __restrict__ p, size_t n16, unsigned long long* sink) {
  uint32_t acc = 0;
  const size_t stride = size_t(gridDim.x) * blockDim.x;
  size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = __ldg(p + i), b = __ldg(p + i + stride), c = __ldg(p + i + 2 * stride), d = __ldg(p + i + 3 * stride);
    acc ^= a.x ^ b.y ^ c.z ^ d.w;
  }
  for (; i < n16; i += stride) acc ^= __ldg(p + i).x;
  if (acc == 0x12345678u) sink[0] = acc;
}

// unit = (slice e, block of 256 rows); per stage two boxes [W bytes x 128 rows]
__global__ void __launch_bounds__(288, 1) ring_kernel(const __grid_constant__ CUtensorMap tm, int E, int row_bytes,
                                                      int W, int S, uint32_t* err, unsigned long long* sink) {
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
  __shared__ RingBars bars;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxS; ++s) {
      mbar_init(&bars.full[s], 1);
      mbar_init(&bars.empty[s], 8);
    }
    bars.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int blocks = 1024 / 256, units = E * blocks, nst = row_bytes / W;
  const uint32_t stage_bytes = 2 * W * 128;
  volatile int* ab = &bars.abort;
  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        const int e = u / blocks, b = u % blocks;
        for (int ss = 0; ss < nst; ++ss, ++it) {
          const int s = it % S;
          if (!bounded_wait(&bars.empty[s], ((it / S) & 1) ^ 1, ab, err)) { ok = false; break; }
          uint8_t* st = sm + s * stage_bytes;
          mbar_arrive_expect_tx(&bars.full[s], stage_bytes);
          tma_load_3d(st, &tm, &bars.full[s], ss * W, b * 256, e);
          tma_load_3d(st + W * 128, &tm, &bars.full[s], ss * W, b * 256 + 128, e);
        }
      }
      // let the copies in flight land before the CTA exits
      const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0;
      for (uint32_t j = first; j < it; ++j) {
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(&bars.full[j % S], (j / S) & 1))
          if (globaltimer() - t0 > kWaitLimitNs) break;
      }
    }
    return;
  }
  uint32_t it = 0;
  unsigned long long acc = 0;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    for (int ss = 0; ss < nst; ++ss, ++it) {
      const int s = it % S;
      if (!bounded_wait(&bars.full[s], (it / S) & 1, ab, err)) return;
      acc += *reinterpret_cast<volatile uint32_t*>(sm + s * stage_bytes + (warp * 32 + lane) * 4);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.empty[s]);
    }
  }
  if (acc == 0x123456789ull) sink[0] = acc;
}

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  const size_t big = size_t(2) << 30, flush_bytes = size_t(512) << 20;
  uint8_t *d, *wflush, *rflush;
  unsigned long long* sink;
  uint32_t* err;
  if (cudaMalloc(&d, big) != cudaSuccess || cudaMalloc(&wflush, flush_bytes) != cudaSuccess ||
      cudaMalloc(&rflush, flush_bytes) != cudaSuccess || cudaMalloc(&sink, 8) != cudaSuccess ||
      cudaMalloc(&err, 64) != cudaSuccess) {
    printf("allocation failed\n");
    return 1;
  }
  cudaMemset(d, 1, big);
  cudaMemset(rflush, 3, flush_bytes);
  cudaMemset(err, 0, 64);
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  auto flush = [&](int mode, int rep) {
    cudaMemsetAsync(wflush, rep, flush_bytes);
    if (mode == 1) read_kernel<<<sms * 2, 512>>>(reinterpret_cast<const uint4*>(rflush), flush_bytes / 16, sink);
  };

  printf("part A: 16-byte loads, %d x 2 CTAs of 512 threads\n", sms);
  for (int mode = 0; mode < 2; ++mode)
    for (size_t mb : {64, 128, 256, 512, 1024, 2048}) {
      const size_t bytes = mb << 20;
      float best = 1e9f;
      for (int rep = 0; rep < 5; ++rep) {
        flush(mode, rep);
        cudaEventRecord(e0);
        read_kernel<<<sms * 2, 512>>>(reinterpret_cast<const uint4*>(d), bytes / 16, sink);
        cudaEventRecord(e1);
        cudaEventSynchronize(e1);
        float ms;
        cudaEventElapsedTime(&ms, e0, e1);
        if (rep > 0 && ms < best) best = ms;
      }
      printf("  %-22s read %5zu MiB: %7.1f us  %5.0f GB/s\n", mode ? "flush write+read" : "flush write only", mb,
             best * 1e3, bytes / (best * 1e-3) / 1e9);
    }

  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", reinterpret_cast<void**>(&enc), 12000,
                                       cudaEnableDefault, &q) != cudaSuccess || !enc) {
    printf("no tensor-map encoder\n");
    return 1;
  }
  const int E = 256, N = 1024, RB = 1024;  // 256 MiB
  const size_t bytes = size_t(E) * N * RB;
  cudaFuncSetAttribute(ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 << 10);
  printf("part B: TMA ring over a [%d][%d][%d B] tensor, clean L2\n", E, N, RB);
  for (int W : {64, 128, 256}) {
    CUtensorMap tm;
    cuuint64_t dims[3] = {(cuuint64_t)RB, (cuuint64_t)N, (cuuint64_t)E};
    cuuint64_t str[2] = {(cuuint64_t)RB, (cuuint64_t)N * RB};
    cuuint32_t box[3] = {(cuuint32_t)W, 128, 1}, es[3] = {1, 1, 1};
    // a 128-byte swizzle needs a 128-byte inner box
    if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, d, dims, str, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            W == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      printf("encode failed W=%d\n", W);
      continue;
    }
    for (int ctas : {1, 2})
      for (int S : {2, 3, 4, 6, 8}) {
        const size_t smem = size_t(S) * 2 * W * 128 + 1024;
        if (smem > (ctas == 1 ? (220u << 10) : (110u << 10))) continue;
        float best = 1e9f;
        for (int rep = 0; rep < 4; ++rep) {
          flush(1, rep);
          cudaEventRecord(e0);
          ring_kernel<<<sms * ctas, 288, smem>>>(tm, E, RB, W, S, err, sink);
          cudaEventRecord(e1);
          cudaEventSynchronize(e1);
          float ms;
          cudaEventElapsedTime(&ms, e0, e1);
          if (rep > 0 && ms < best) best = ms;
        }
        unsigned herr = 0;
        cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost);
        printf("  box %3d B x 128 rows, %d CTA/SM, %d stages (%6zu B in flight per SM): %6.1f us  %5.0f GB/s%s\n", W,
               ctas, S, size_t(ctas) * S * 2 * W * 128, best * 1e3, bytes / (best * 1e-3) / 1e9,
               herr ? "  (timeout)" : "");
      }
  }
  const cudaError_t ce = cudaDeviceSynchronize();
  printf("%s\n", cudaGetErrorString(ce));
  return ce == cudaSuccess ? 0 : 1;
}
