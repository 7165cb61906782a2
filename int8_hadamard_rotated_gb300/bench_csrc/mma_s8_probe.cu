// mma_s8_probe.cu -- a microbenchmark of the legacy 8-bit integer tensor path
// (mma.sync m16n8k32 s8 x s8 -> s32), built into the benchmark's own small
// library (libconvrot_bench.so), not into libconvrot.so. It gives the GEMM's
// roofline its context: sm_103a's tcgen05 tensor cores have no 8-bit integer
// kind, so the exact INT8 product runs on binary16 operands; this measures
// what the only INT8 tensor instruction left would deliver. Not part of the
// method.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeChains = 8;  // independent accumulators per warp

// Every warp issues `iters` rounds of kProbeChains independent m16n8k32 MMAs on
// register operands (no memory traffic); the sums feed a data-dependent store
// that never happens for these inputs, so the work is not removed.
__global__ void __launch_bounds__(kProbeThreads) mma_s8_probe_kernel(int iters, int* sink) {
  const uint32_t lane = threadIdx.x & 31;
  uint32_t a[4], b[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) a[i] = 0x01010101u * ((lane + i) & 3);
  b[0] = 0x01010101u * (lane & 1);
  b[1] = 0x01010101u * ((lane >> 1) & 1);
  int acc[kProbeChains][4];
#pragma unroll
  for (int c = 0; c < kProbeChains; ++c)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[c][i] = 0;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < kProbeChains; ++c) {
      asm volatile(
          "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
          "{%0, %1, %2, %3};"
          : "+r"(acc[c][0]), "+r"(acc[c][1]), "+r"(acc[c][2]), "+r"(acc[c][3])
          : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
    }
  }
  int s = 0;
#pragma unroll
  for (int c = 0; c < kProbeChains; ++c) s += acc[c][0] ^ acc[c][1] ^ acc[c][2] ^ acc[c][3];
  if (s == 0x7fffffff) atomicAdd(sink, 1);
}

}  // namespace

// Returns 0 and the rate in *tops (tera-ops per second, two per multiply-add),
// 1 for bad arguments, 2 if the current device is not sm_103, or 3 + the
// cudaError_t of a failed CUDA call. Synchronous; allocates 4 bytes.
extern "C" int bench_probe_int8_mma_rate(int iters, double* tops) {
  if (iters <= 0 || !tops) return 1;
  int dev = 0;
  cudaDeviceProp prop;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return 3;
  if (prop.major != 10 || prop.minor != 3) return 2;
  int* sink = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  int st = 0;
  const int blocks = prop.multiProcessorCount * 4;
  float ms = 0.0f;
  if (cudaMalloc(&sink, sizeof(int)) != cudaSuccess || cudaEventCreate(&e0) != cudaSuccess ||
      cudaEventCreate(&e1) != cudaSuccess) {
    st = 3 + static_cast<int>(cudaGetLastError());
  } else {
    mma_s8_probe_kernel<<<blocks, kProbeThreads>>>(iters / 10 + 1, sink);  // warm-up
    cudaEventRecord(e0);
    mma_s8_probe_kernel<<<blocks, kProbeThreads>>>(iters, sink);
    cudaEventRecord(e1);
    const cudaError_t e = cudaEventSynchronize(e1);
    if (e != cudaSuccess) st = 3 + static_cast<int>(e);
    else if (cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess || ms <= 0.0f) st = 3 + static_cast<int>(cudaErrorUnknown);
  }
  if (st == 0) {
    const double ops = 2.0 * 16 * 8 * 32 * kProbeChains * static_cast<double>(iters) * blocks * (kProbeThreads / 32);
    *tops = ops / (ms * 1e-3) / 1e12;
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (sink) cudaFree(sink);
  return st;
}
