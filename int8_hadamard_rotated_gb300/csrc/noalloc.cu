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
// The address is remembered together with the identity of the CUDA context
// it was looked up in; a call made in another context (for instance after
// cudaDeviceReset replaced the device's primary context) looks it up again,
// so no call ever uses an address of a context that no longer exists. The
// first call on a device (or in a new context) should therefore come before
// any stream capture.
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
struct ScratchAddr {
  unsigned long long ctx_id = 0;  // the context the address belongs to (0: none yet)
  void* addr = nullptr;
};
ScratchAddr g_scratch_addr[kMaxDevices];  // per device

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current CUDA context (0 if there is none).
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the array in the current device's current context,
// looked up on the first call in that context.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return CONVROT_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchAddr& a = g_scratch_addr[dev];
  const unsigned long long ctx = current_context_id();
  if (ctx == 0 || ctx != a.ctx_id || !a.addr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // makes the device's context current if needed
    if (e != cudaSuccess) return set_cuda_error(e);
    if (!p) return set_cuda_error(cudaErrorInvalidSymbol);
    a.addr = p;
    a.ctx_id = current_context_id();
  }
  *out = a.addr;
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
