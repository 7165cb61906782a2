// copy_ceiling.cu -- the benchmark's size-matched streaming copy, built into
// libconvrot_bench.so (not into libconvrot.so). It moves exactly the bytes of
// a pack launch, with none of the pack's arithmetic: it reads fp32 rows
// [M, K], writes one byte (or two) per element, converted by truncation, and
// one fp32 word per row. Timed under the same protocol as the pack (L2
// flushed before the launch, CUDA events on the launching stream), it is the
// bandwidth a kernel with the pack's traffic can reach on this GPU, the
// ceiling the pack's HBM fraction is read against. Not part of the method.
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace {

constexpr int kThreads = 256;
constexpr int kVec = 4;  // 16-byte input vectors in flight per thread per round

// Element e of X (fp32) -> byte (or binary16) e of out; row r's word -> scales[r].
template <int OSZ>
__global__ void __launch_bounds__(kThreads) copy_ceiling_kernel(const float4* __restrict__ x, int64_t n4,
                                                                 void* __restrict__ out, float* __restrict__ scales,
                                                                 int64_t M) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  for (; i + (kVec - 1) * stride < n4; i += kVec * stride) {
    float4 v[kVec];
#pragma unroll
    for (int k = 0; k < kVec; ++k) v[k] = __ldcs(x + i + k * stride);
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      if (OSZ == 1) {
        const uint32_t w = (static_cast<uint32_t>(static_cast<int>(v[k].x)) & 0xffu) |
                           ((static_cast<uint32_t>(static_cast<int>(v[k].y)) & 0xffu) << 8) |
                           ((static_cast<uint32_t>(static_cast<int>(v[k].z)) & 0xffu) << 16) |
                           (static_cast<uint32_t>(static_cast<int>(v[k].w)) << 24);
        reinterpret_cast<uint32_t*>(out)[i + k * stride] = w;
      } else {
        __half2 a = __floats2half2_rn(v[k].x, v[k].y), b = __floats2half2_rn(v[k].z, v[k].w);
        uint2 w;
        w.x = *reinterpret_cast<uint32_t*>(&a);
        w.y = *reinterpret_cast<uint32_t*>(&b);
        reinterpret_cast<uint2*>(out)[i + k * stride] = w;
      }
    }
  }
  for (; i < n4; i += stride) {
    const float4 v = __ldcs(x + i);
    if (OSZ == 1) {
      const uint32_t w = (static_cast<uint32_t>(static_cast<int>(v.x)) & 0xffu) |
                         ((static_cast<uint32_t>(static_cast<int>(v.y)) & 0xffu) << 8) |
                         ((static_cast<uint32_t>(static_cast<int>(v.z)) & 0xffu) << 16) |
                         (static_cast<uint32_t>(static_cast<int>(v.w)) << 24);
      reinterpret_cast<uint32_t*>(out)[i] = w;
    } else {
      __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
      uint2 w;
      w.x = *reinterpret_cast<uint32_t*>(&a);
      w.y = *reinterpret_cast<uint32_t*>(&b);
      reinterpret_cast<uint2*>(out)[i] = w;
    }
  }
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  for (int64_t r = t; r < M; r += stride) scales[r] = 0.0f;
}

}  // namespace

// X fp32 [M, K] (16-byte aligned, K % 4 == 0) -> out [M, K] of out_bytes (1 or
// 2) per element, scales [M]; grid = ctas_per_sm x SMs. Returns 0, 1 for bad
// arguments, or 3 + the cudaError_t of a failed launch.
extern "C" int bench_copy_ceiling(const void* X, int64_t M, int64_t K, int out_bytes, void* out, float* scales,
                                  int ctas_per_sm, void* stream) {
  if (!X || !out || !scales || M < 0 || K <= 0 || K % 4 != 0 || (out_bytes != 1 && out_bytes != 2) ||
      ctas_per_sm <= 0)
    return 1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 3;
  const int64_t n4 = M * K / 4;
  const unsigned grid = static_cast<unsigned>(sms * ctas_per_sm);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (out_bytes == 1)
    copy_ceiling_kernel<1><<<grid, kThreads, 0, s>>>(static_cast<const float4*>(X), n4, out, scales, M);
  else
    copy_ceiling_kernel<2><<<grid, kThreads, 0, s>>>(static_cast<const float4*>(X), n4, out, scales, M);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? 0 : 3 + static_cast<int>(e);
}
