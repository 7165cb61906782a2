// noalloc.cu -- convrot_linear_noalloc: the fused convrot linear for callers
// that cannot allocate device memory.
//
// convrot_linear needs a caller-provided workspace for the packed activation
// (binary16 codes and row scales). Some callers have no way to provide one: a
// plugin that a host framework hands only its input and output buffers while
// the framework owns every allocation, or a latency-bound loop where
// cudaMalloc is not allowed because it can synchronize the device and take
// milliseconds. This entry point keeps the packed activation in a fixed array
// owned by the library instead, so such a caller passes only its inputs and
// outputs.
//
// The array is a file-scope __device__ variable of CONVROT_NOALLOC_SCRATCH_BYTES
// bytes: every GPU that loads this library holds it until the process exits.
// In host code its name is a host-side stand-in, not a device address, so its
// device address is looked up with cudaGetSymbolAddress, with that device
// current, by the first call on each device, and then passed to the kernels.
// That first call on a device should therefore come before any stream capture.
// All calls on a device share the array and it keeps the last call's
// contents; nothing in it needs to start at zero, because the pack writes
// every code and scale that the GEMM then reads. Calls that overlap on the
// GPU (on different streams, or from host threads racing on one device) race
// on the array.
#include "common.cuh"

#include <mutex>

namespace convrot {
namespace {

constexpr size_t kScratchBytes = CONVROT_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The packed activation of convrot_linear_noalloc: [M,K] binary16 codes, then
// (at the next 256-byte boundary) [M] fp32 row scales.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];  // device address of the array, per device

// Device address of the array on the current device, looked up on the first
// call for that device.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return CONVROT_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return set_cuda_error(e);
    if (!p) return set_cuda_error(cudaErrorInvalidSymbol);
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return CONVROT_OK;
}

}  // namespace
}  // namespace convrot

using namespace convrot;

extern "C" int convrot_linear_noalloc(const void* X, int x_dtype, int64_t M, int64_t K, int G,
                                      const convrot_weight* weights, int n_weights, void* stream) {
  if (M < 0 || K <= 0) return CONVROT_ERR_ARG;
  if (x_dtype != CONVROT_F32 && x_dtype != CONVROT_F16) return CONVROT_ERR_ARG;
  if (int st = check_weight_list(weights, n_weights)) return st;
  if (M == 0) return CONVROT_OK;
  if (!X) return CONVROT_ERR_ARG;
  if (!valid_group(G, K)) return CONVROT_ERR_GROUP;
  if (K % 16 != 0 || !aligned16(X)) return CONVROT_ERR_ALIGN;
  if (K > CONVROT_PACK_MAX_K) return CONVROT_ERR_UNSUPPORTED;
  if (M > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
  const size_t codes_bytes = round256(static_cast<size_t>(M) * K * 2);
  const size_t need = codes_bytes + round256(static_cast<size_t>(M) * 4);
  if (need > kScratchBytes) return CONVROT_ERR_SCRATCH;
  const size_t esz = x_dtype == CONVROT_F32 ? 4 : 2;
  const size_t nx = static_cast<size_t>(M) * K * esz;
  if (int st = check_weights(weights, n_weights, M, K, X, nx, nullptr, 0)) return st;
  if (int st = check_device()) return st;
  void* base = nullptr;
  if (int st = scratch_address(&base)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(base);
  __half* x16 = reinterpret_cast<__half*>(ws);
  float* s_x = reinterpret_cast<float*>(ws + codes_bytes);
  int st = launch_pack(X, x_dtype, M, K, G, x16, kPackF16, s_x, s);
  if (st) return st;
  return launch_grouped(x16, s_x, M, K, weights, n_weights, s);
}
