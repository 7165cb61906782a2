// api.cu -- the extern "C" entry points of libconvrot.so (see include/convrot.h).
//
// Each entry point checks its arguments on the host (sizes, group rule,
// alignment, int32 overflow bound, aliasing, workspace size), then enqueues
// the kernels on the caller's stream. No entry point allocates device memory.
#include "common.cuh"

#include <cstring>
#include <mutex>

namespace convrot {

namespace {
thread_local int t_last_cuda_error = 0;

struct DevInfo {
  int sm_count = 0;
  int is_sm103 = -1;  // -1 unknown
};
std::mutex g_dev_mu;
DevInfo g_dev[64];

DevInfo* dev_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (d.is_sm103 < 0) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return nullptr;
    d.sm_count = prop.multiProcessorCount;
    d.is_sm103 = (prop.major == 10 && prop.minor == 3) ? 1 : 0;
  }
  return &d;
}
}  // namespace

int set_cuda_error(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return CONVROT_ERR_CUDA;
}

int check_launch() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CONVROT_OK : set_cuda_error(e);
}

int device_sm_count() {
  DevInfo* d = dev_info();
  return (d && d->sm_count > 0) ? d->sm_count : 1;
}

bool device_is_sm103() {
  DevInfo* d = dev_info();
  return d && d->is_sm103 == 1;
}

int read_and_clear_device_error(cudaStream_t stream);  // gemm.cu: syncs, then the GEMM's word
int read_and_clear_w4_error();                         // gemm_w4.cu: the S8 x S4 GEMM's word
int read_and_clear_pack_error();                       // pack.cu: the pack kernels' word

}  // namespace convrot

namespace convrot {

bool valid_group(int G, int64_t K) {
  if (G < 1 || G > 1024) return false;
  int g = G;
  while (g % 4 == 0) g /= 4;
  return g == 1 && K % G == 0;
}

size_t round256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

int check_device() { return device_is_sm103() ? CONVROT_OK : CONVROT_ERR_DEVICE; }

}  // namespace convrot

using namespace convrot;

namespace {

int pack_checks(const void* X, int x_dtype, int64_t M, int64_t K, int G, const void* Q, size_t q_esz,
                const float* s);

}  // namespace

extern "C" {

int convrot_version(void) { return 100; }

const char* convrot_strerror(int status) {
  switch (status) {
    case CONVROT_OK: return "ok";
    case CONVROT_ERR_ARG: return "invalid argument (null array, negative size, unknown dtype or linear count)";
    case CONVROT_ERR_GROUP: return "group size must be 4^n in [1,1024] and divide K";
    case CONVROT_ERR_ALIGN: return "arrays must be 16-byte aligned and K a multiple of 16";
    case CONVROT_ERR_OVERFLOW: return "K too large: int32 accumulation could overflow (K > 133144)";
    case CONVROT_ERR_ALIAS: return "an output overlaps an input or another output";
    case CONVROT_ERR_WORKSPACE: return "workspace missing or too small";
    case CONVROT_ERR_UNSUPPORTED: return "shape beyond this build's limits";
    case CONVROT_ERR_TIMEOUT: return "a device-side wait timed out";
    case CONVROT_ERR_CUDA: return "CUDA runtime error";
    case CONVROT_ERR_DEVICE: return "the current device is not an sm_103 GPU";
    case CONVROT_ERR_SCRATCH: return "packed activation larger than the fixed scratch (CONVROT_NOALLOC_SCRATCH_BYTES)";
    default: return "unknown status";
  }
}

int convrot_last_cuda_error(void) { return t_last_cuda_error; }

int convrot_pack_activations(const void* X, int x_dtype, int64_t M, int64_t K, int G,
                             int8_t* Q_x, float* s_x, void* stream) {
  if (int st = pack_checks(X, x_dtype, M, K, G, Q_x, 1, s_x)) return st;
  if (M == 0) return CONVROT_OK;
  return launch_pack(X, x_dtype, M, K, G, Q_x, kPackI8, s_x, static_cast<cudaStream_t>(stream));
}

int convrot_prepare_weight(const float* W, int64_t N, int64_t K, int G,
                           int8_t* Q_w, float* s_w, uint16_t* Q_w16, void* stream) {
  if (N < 0 || K <= 0) return CONVROT_ERR_ARG;
  if (N == 0) return CONVROT_OK;
  if (!W || !Q_w || !s_w) return CONVROT_ERR_ARG;
  if (!valid_group(G, K)) return CONVROT_ERR_GROUP;
  if (K % 16 != 0 || !aligned16(W) || !aligned16(Q_w) || !aligned16(s_w) || (Q_w16 && !aligned16(Q_w16)))
    return CONVROT_ERR_ALIGN;
  if (K > CONVROT_PACK_MAX_K) return CONVROT_ERR_UNSUPPORTED;
  const size_t nw = static_cast<size_t>(N) * K * 4, nq = static_cast<size_t>(N) * K, ns = static_cast<size_t>(N) * 4;
  const size_t nh = static_cast<size_t>(N) * K * 2;
  if (overlaps(W, nw, Q_w, nq) || overlaps(W, nw, s_w, ns) || overlaps(Q_w, nq, s_w, ns) ||
      overlaps(Q_w16, nh, W, nw) || overlaps(Q_w16, nh, Q_w, nq) || overlaps(Q_w16, nh, s_w, ns))
    return CONVROT_ERR_ALIAS;
  if (int st = check_device()) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int st = launch_pack(W, CONVROT_F32, N, K, G, Q_w, kPackI8, s_w, s);
  if (st == CONVROT_OK && Q_w16) st = launch_widen(Q_w, reinterpret_cast<__half*>(Q_w16), N * K, s);
  return st;
}

size_t int8_linear_workspace_size(int64_t M, int64_t N, int64_t K, int have_q_w16) {
  if (M < 0 || N < 0 || K < 0) return 0;
  size_t b = round256(static_cast<size_t>(M) * K * 2);
  if (!have_q_w16) b += round256(static_cast<size_t>(N) * K * 2);
  return b + CONVROT_GEMM_SYNC_BYTES;
}

size_t convrot_linear_workspace_size(int64_t M, int64_t K) {
  if (M < 0 || K < 0) return 0;
  return round256(static_cast<size_t>(M) * K * 2) + round256(static_cast<size_t>(M) * 4) +
         CONVROT_GEMM_SYNC_BYTES;
}

}  // extern "C"

namespace {

// Shared checks and workspace carving of int8_linear / int8_gemm_s32.
int int8_gemm_common(const int8_t* Q_x, const float* s_x, int64_t M, int64_t K,
                     const int8_t* Q_w, const uint16_t* Q_w16, const int32_t* kchunk, const float* s_w,
                     const float* bias, int64_t N, void* out, size_t out_esz, bool raw,
                     void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 0 || N < 0 || K <= 0) return CONVROT_ERR_ARG;
  if (M == 0 || N == 0) return CONVROT_OK;
  if (!Q_x || (!raw && !s_x) || (!Q_w && !Q_w16) || !out) return CONVROT_ERR_ARG;
  if (M > 0x7fffffff || N > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
  if (K % 16 != 0 || !aligned16(Q_x) || !aligned16(out) || (s_x && !aligned16(s_x)) ||
      (Q_w && !aligned16(Q_w)) || (Q_w16 && !aligned16(Q_w16)) || (s_w && !aligned16(s_w)) ||
      (bias && !aligned16(bias)) || (workspace && !aligned16(workspace)) ||
      (reinterpret_cast<uintptr_t>(kchunk) & 3u))
    return CONVROT_ERR_ALIGN;
  if (K > CONVROT_MAX_K) return CONVROT_ERR_OVERFLOW;
  const size_t need = int8_linear_workspace_size(M, N, K, Q_w16 != nullptr);
  if (!workspace || workspace_bytes < need) return CONVROT_ERR_WORKSPACE;
  const size_t no = static_cast<size_t>(M) * N * out_esz;
  const size_t mk = static_cast<size_t>(M) * K, nk = static_cast<size_t>(N) * K;
  if (overlaps(out, no, Q_x, mk) || overlaps(out, no, s_x, M * 4) || overlaps(out, no, Q_w, nk) ||
      overlaps(out, no, Q_w16, nk * 2) || overlaps(out, no, s_w, N * 4) || overlaps(out, no, bias, N * 4) ||
      overlaps(out, no, workspace, need))
    return CONVROT_ERR_ALIAS;
  if (overlaps(workspace, need, Q_x, mk) || overlaps(workspace, need, s_x, M * 4) ||
      overlaps(workspace, need, Q_w, nk) || overlaps(workspace, need, Q_w16, nk * 2) ||
      overlaps(workspace, need, s_w, N * 4) || overlaps(workspace, need, bias, N * 4))
    return CONVROT_ERR_ALIAS;
  if (int st = check_device()) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __half* x16 = reinterpret_cast<__half*>(ws);
  const __half* w16 = reinterpret_cast<const __half*>(Q_w16);
  int st = launch_widen(Q_x, x16, M * K, s);
  if (st) return st;
  if (!w16) {
    __half* wtmp = reinterpret_cast<__half*>(ws + round256(mk * 2));
    st = launch_widen(Q_w, wtmp, N * K, s);
    if (st) return st;
    w16 = wtmp;
  }
  GemmLinear lin{w16, s_w, bias, out, N, kchunk};
  return launch_gemm(x16, s_x, M, K, &lin, 1, raw, s, sync_at(ws + need - CONVROT_GEMM_SYNC_BYTES));
}

}  // namespace

extern "C" {

int int8_linear(const int8_t* Q_x, const float* s_x, int64_t M, int64_t K,
                const int8_t* Q_w, const uint16_t* Q_w16, const float* s_w,
                const float* bias, int64_t N, float* Y,
                void* workspace, size_t workspace_bytes, void* stream) {
  return int8_gemm_common(Q_x, s_x, M, K, Q_w, Q_w16, nullptr, s_w, bias, N, Y, 4, false,
                          workspace, workspace_bytes, stream);
}

int int8_gemm_s32(const int8_t* Q_x, int64_t M, int64_t K,
                  const int8_t* Q_w, const uint16_t* Q_w16, const int32_t* kchunk, int64_t N,
                  int32_t* A, void* workspace, size_t workspace_bytes, void* stream) {
  return int8_gemm_common(Q_x, nullptr, M, K, Q_w, Q_w16, kchunk, nullptr, nullptr, N, A, 4, true,
                          workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace convrot {

// Checks of the weight descriptors against each other and against the
// activation-side arrays [in0, in0+n0) and [in1, in1+n1).
int check_weights(const convrot_weight* weights, int n_weights, int64_t M, int64_t K,
                  const void* in0, size_t n0, const void* in1, size_t n1) {
  for (int j = 0; j < n_weights; ++j) {
    const convrot_weight& w = weights[j];
    if (w.N == 0) continue;
    if (!aligned16(weight_codes(w)) || !aligned16(w.Y) || (w.scale && !aligned16(w.scale)) ||
        (w.bias && !aligned16(w.bias)) || (reinterpret_cast<uintptr_t>(w.kchunk) & 3u))
      return CONVROT_ERR_ALIGN;
    if (w.q4) {
      // the S8 x S4 GEMM: 64-value blocks of K, whole 16-byte rows of Y, one exact fp32 run
      if (K % 64 != 0 || w.N % 4 != 0) return CONVROT_ERR_ALIGN;
      if (K > CONVROT_W4_MAX_K) return CONVROT_ERR_UNSUPPORTED;
    }
  }
  for (int j = 0; j < n_weights; ++j) {
    const convrot_weight& w = weights[j];
    if (w.N == 0) continue;
    if (w.N > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
    const size_t ny = static_cast<size_t>(M) * w.N * 4, nk = weight_code_bytes(w, K);
    const void* wk = weight_codes(w);
    if (overlaps(w.Y, ny, in0, n0) || overlaps(w.Y, ny, in1, n1)) return CONVROT_ERR_ALIAS;
    if (overlaps(in0, n0, wk, nk) || overlaps(in1, n1, wk, nk)) return CONVROT_ERR_ALIAS;
    for (int i = 0; i < n_weights; ++i) {
      const convrot_weight& v = weights[i];
      if (v.N == 0) continue;
      const size_t vk = weight_code_bytes(v, K);
      if (overlaps(w.Y, ny, weight_codes(v), vk) || overlaps(w.Y, ny, v.scale, v.N * 4) ||
          overlaps(w.Y, ny, v.bias, v.N * 4))
        return CONVROT_ERR_ALIAS;
      if (i != j && overlaps(w.Y, ny, v.Y, static_cast<size_t>(M) * v.N * 4)) return CONVROT_ERR_ALIAS;
    }
  }
  return CONVROT_OK;
}

int check_weight_list(const convrot_weight* weights, int n_weights) {
  if (!weights || n_weights < 1 || n_weights > CONVROT_MAX_LINEARS) return CONVROT_ERR_ARG;
  for (int j = 0; j < n_weights; ++j) {
    const convrot_weight& w = weights[j];
    if (w.N < 0) return CONVROT_ERR_ARG;
    if (w.N > 0 && (!w.Y || (!w.q16) == (!w.q4))) return CONVROT_ERR_ARG;  // exactly one kind of weight
  }
  return CONVROT_OK;
}

int launch_linears(const __half* x16, const float* s_x, int64_t M, int64_t K, const GemmLinear* lins, int n_lin,
                   bool raw_s32, cudaStream_t s, GemmSync sync) {
  GemmLinear w16[CONVROT_MAX_LINEARS], w4[CONVROT_MAX_LINEARS];
  int n16 = 0, n4 = 0;
  for (int j = 0; j < n_lin; ++j) {
    if (lins[j].N == 0) continue;
    if (lins[j].w16) w16[n16++] = lins[j];
    else w4[n4++] = lins[j];
  }
  if (n16 > 0)
    if (int st = launch_gemm(x16, s_x, M, K, w16, n16, raw_s32, s, sync)) return st;
  if (n4 > 0) return launch_gemm_w4(x16, s_x, M, K, w4, n4, raw_s32, s, sync);
  return CONVROT_OK;
}

int launch_grouped(const __half* x16, const float* s_x, int64_t M, int64_t K,
                   const convrot_weight* weights, int n_weights, cudaStream_t s, float in_scale,
                   GemmSync sync) {
  GemmLinear lins[CONVROT_MAX_LINEARS];
  int n = 0;
  for (int j = 0; j < n_weights; ++j) {
    const convrot_weight& w = weights[j];
    if (w.N == 0) continue;
    lins[n++] = to_linear(w, w.Y, in_scale);
  }
  if (n == 0) return CONVROT_OK;
  return launch_linears(x16, s_x, M, K, lins, n, false, s, sync);
}

}  // namespace convrot

namespace {

int pack_checks(const void* X, int x_dtype, int64_t M, int64_t K, int G, const void* Q, size_t q_esz,
                const float* s) {
  if (M < 0 || K <= 0) return CONVROT_ERR_ARG;
  if (x_dtype != CONVROT_F32 && x_dtype != CONVROT_F16) return CONVROT_ERR_ARG;
  if (M == 0) return CONVROT_OK;
  if (!X || !Q || !s) return CONVROT_ERR_ARG;
  if (!valid_group(G, K)) return CONVROT_ERR_GROUP;
  if (K % 16 != 0 || !aligned16(X) || !aligned16(Q) || !aligned16(s)) return CONVROT_ERR_ALIGN;
  if (K > CONVROT_PACK_MAX_K) return CONVROT_ERR_UNSUPPORTED;
  if (M > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
  const size_t esz = x_dtype == CONVROT_F32 ? 4 : 2;
  const size_t nx = static_cast<size_t>(M) * K * esz, nq = static_cast<size_t>(M) * K * q_esz,
               ns = static_cast<size_t>(M) * 4;
  if (overlaps(X, nx, Q, nq) || overlaps(X, nx, s, ns) || overlaps(Q, nq, s, ns)) return CONVROT_ERR_ALIAS;
  return check_device();
}

}  // namespace

extern "C" {

int convrot_pack_activations_f16(const void* X, int x_dtype, int64_t M, int64_t K,
                                 int G, uint16_t* Q_x16, float* s_x, void* stream) {
  if (int st = pack_checks(X, x_dtype, M, K, G, Q_x16, 2, s_x)) return st;
  if (M == 0) return CONVROT_OK;
  return launch_pack(X, x_dtype, M, K, G, Q_x16, kPackF16, s_x, static_cast<cudaStream_t>(stream));
}

int convrot_pack_gelu_f16(const float* X, int64_t M, int64_t K, int G, uint16_t* Q_x16, float* s_x, void* stream) {
  if (int st = pack_checks(X, CONVROT_F32, M, K, G, Q_x16, 2, s_x)) return st;
  if (M == 0) return CONVROT_OK;
  return launch_pack_gelu(X, M, K, G, reinterpret_cast<__half*>(Q_x16), s_x, static_cast<cudaStream_t>(stream));
}

int convrot_linear_packed(const uint16_t* Q_x16, const float* s_x, int64_t M, int64_t K,
                          const convrot_weight* weights, int n_weights,
                          void* workspace, size_t workspace_bytes, void* stream) {
  return convrot_linear_packed_act(Q_x16, s_x, M, K, weights, n_weights, CONVROT_ACT_NONE, workspace,
                                   workspace_bytes, stream);
}

int convrot_linear_packed_act(const uint16_t* Q_x16, const float* s_x, int64_t M, int64_t K,
                              const convrot_weight* weights, int n_weights, int activation,
                              void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 0 || K <= 0) return CONVROT_ERR_ARG;
  if (activation != CONVROT_ACT_NONE && activation != CONVROT_ACT_GELU && activation != CONVROT_ACT_SWIGLU)
    return CONVROT_ERR_ARG;
  if (int st = check_weight_list(weights, n_weights)) return st;
  const bool swiglu = (activation == CONVROT_ACT_SWIGLU);
  if (swiglu && (n_weights != 2 || weights[1].N != weights[0].N || weights[0].N == 0)) return CONVROT_ERR_ARG;
  if (swiglu && (!weights[0].q16 || !weights[1].q16)) return CONVROT_ERR_UNSUPPORTED;
  if (M == 0) return CONVROT_OK;
  if (!Q_x16 || !s_x) return CONVROT_ERR_ARG;
  if (K % 16 != 0 || !aligned16(Q_x16) || !aligned16(s_x) || (workspace && !aligned16(workspace)))
    return CONVROT_ERR_ALIGN;
  if (workspace && workspace_bytes < CONVROT_GEMM_SYNC_BYTES) return CONVROT_ERR_WORKSPACE;
  if (K > CONVROT_MAX_K) return CONVROT_ERR_OVERFLOW;
  if (M > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
  if (workspace && (overlaps(workspace, CONVROT_GEMM_SYNC_BYTES, Q_x16, static_cast<size_t>(M) * K * 2) ||
                    overlaps(workspace, CONVROT_GEMM_SYNC_BYTES, s_x, static_cast<size_t>(M) * 4)))
    return CONVROT_ERR_ALIAS;
  // split SwiGLU: both descriptors write h to the first one's Y, so each is
  // checked on its own, then h against the other weight's arrays
  convrot_weight w2[2];
  const convrot_weight* ws_list = weights;
  if (swiglu) {
    w2[0] = weights[0];
    w2[1] = weights[1];
    w2[1].Y = w2[0].Y;
    ws_list = w2;
    for (int j = 0; j < 2; ++j)
      if (int st = check_weights(&w2[j], 1, M, K, Q_x16, static_cast<size_t>(M) * K * 2, s_x,
                                 static_cast<size_t>(M) * 4))
        return st;
    const size_t ny = static_cast<size_t>(M) * w2[0].N * 4;
    for (int j = 0; j < 2; ++j)
      if (overlaps(w2[0].Y, ny, weight_codes(w2[j]), weight_code_bytes(w2[j], K)) ||
          overlaps(w2[0].Y, ny, w2[j].scale, w2[j].N * 4) || overlaps(w2[0].Y, ny, w2[j].bias, w2[j].N * 4))
        return CONVROT_ERR_ALIAS;
  } else if (int st = check_weights(weights, n_weights, M, K, Q_x16, static_cast<size_t>(M) * K * 2, s_x,
                                    static_cast<size_t>(M) * 4)) {
    return st;
  }
  if (workspace)
    for (int j = 0; j < n_weights; ++j) {
      const convrot_weight& w = ws_list[j];
      if (w.N == 0) continue;
      if (overlaps(workspace, CONVROT_GEMM_SYNC_BYTES, w.Y, static_cast<size_t>(M) * w.N * 4) ||
          overlaps(workspace, CONVROT_GEMM_SYNC_BYTES, weight_codes(w), weight_code_bytes(w, K)) ||
          (w.scale && overlaps(workspace, CONVROT_GEMM_SYNC_BYTES, w.scale, w.N * 4)) ||
          (w.bias && overlaps(workspace, CONVROT_GEMM_SYNC_BYTES, w.bias, w.N * 4)))
        return CONVROT_ERR_ALIAS;
    }
  if (int st = check_device()) return st;
  const GemmSync sync = workspace ? sync_at(workspace) : GemmSync();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const __half* x16 = reinterpret_cast<const __half*>(Q_x16);
  if (activation == CONVROT_ACT_NONE) return launch_grouped(x16, s_x, M, K, weights, n_weights, s, 1.0f, sync);
  GemmLinear lins[CONVROT_MAX_LINEARS];
  int n = 0;
  for (int j = 0; j < n_weights; ++j)
    if (ws_list[j].N > 0) lins[n++] = to_linear(ws_list[j], ws_list[j].Y);
  return launch_gemm_act(x16, s_x, M, K, lins, n, activation, s, sync);
}

int convrot_test_handover_timeout(const uint16_t* Q_x16, const float* s_x, int64_t M, int64_t K,
                                  const convrot_weight* weights, int n_weights, void* workspace,
                                  size_t workspace_bytes, uint64_t wait_ns, void* stream) {
  if (M <= 0 || K <= 0 || wait_ns == 0) return CONVROT_ERR_ARG;
  if (int st = check_weight_list(weights, n_weights)) return st;
  for (int j = 0; j < n_weights; ++j)
    if (weights[j].q4) return CONVROT_ERR_ARG;  // the binary16-weight GEMM
  if (!Q_x16 || !s_x || !workspace) return CONVROT_ERR_ARG;
  if (K % 16 != 0 || !aligned16(Q_x16) || !aligned16(s_x) || !aligned16(workspace)) return CONVROT_ERR_ALIGN;
  if (workspace_bytes < CONVROT_GEMM_SYNC_BYTES) return CONVROT_ERR_WORKSPACE;
  if (K > CONVROT_MAX_K) return CONVROT_ERR_OVERFLOW;
  if (M > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
  if (int st = check_weights(weights, n_weights, M, K, Q_x16, static_cast<size_t>(M) * K * 2, s_x,
                             static_cast<size_t>(M) * 4))
    return st;
  if (int st = check_device()) return st;
  GemmSync sync = sync_at(workspace);
  sync.test_wait_ns = wait_ns;
  sync.test_unpublished_handover = true;
  return launch_grouped(reinterpret_cast<const __half*>(Q_x16), s_x, M, K, weights, n_weights,
                        static_cast<cudaStream_t>(stream), 1.0f, sync);
}

int convrot_test_unscale_sweep(const float* divisors, int n_divisors, int y_exp, uint64_t* mismatches,
                               uint64_t* first, void* stream) {
  if (!divisors || !mismatches || !first || n_divisors < 1 || n_divisors > 65535) return CONVROT_ERR_ARG;
  if (y_exp < -98 || y_exp > 97) return CONVROT_ERR_ARG;  // inside the step's range
  if (!aligned16(divisors) || reinterpret_cast<uintptr_t>(mismatches) % 8 != 0 ||
      reinterpret_cast<uintptr_t>(first) % 8 != 0)
    return CONVROT_ERR_ALIGN;
  if (int st = check_device()) return st;
  return launch_unscale_sweep(divisors, n_divisors, y_exp, reinterpret_cast<unsigned long long*>(mismatches),
                              reinterpret_cast<unsigned long long*>(first), static_cast<cudaStream_t>(stream));
}

int convrot_linear(const void* X, int x_dtype, int64_t M, int64_t K, int G,
                   const convrot_weight* weights, int n_weights,
                   void* workspace, size_t workspace_bytes, void* stream) {
  return convrot_linear_scaled(X, x_dtype, M, K, G, 1.0f, weights, n_weights, workspace, workspace_bytes,
                               stream);
}

int convrot_linear_scaled(const void* X, int x_dtype, int64_t M, int64_t K, int G, float input_scale,
                          const convrot_weight* weights, int n_weights,
                          void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 0 || K <= 0) return CONVROT_ERR_ARG;
  if (!(input_scale > 0.0f) || !(input_scale <= 3.402823466e38f)) return CONVROT_ERR_ARG;  // finite, > 0
  if (x_dtype != CONVROT_F32 && x_dtype != CONVROT_F16) return CONVROT_ERR_ARG;
  if (int st = check_weight_list(weights, n_weights)) return st;
  if (M == 0) return CONVROT_OK;
  if (!X) return CONVROT_ERR_ARG;
  if (!valid_group(G, K)) return CONVROT_ERR_GROUP;
  if (K % 16 != 0 || !aligned16(X) || (workspace && !aligned16(workspace))) return CONVROT_ERR_ALIGN;
  if (K > CONVROT_PACK_MAX_K) return CONVROT_ERR_UNSUPPORTED;
  if (M > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
  const size_t need = convrot_linear_workspace_size(M, K);
  if (!workspace || workspace_bytes < need) return CONVROT_ERR_WORKSPACE;
  const size_t esz = x_dtype == CONVROT_F32 ? 4 : 2;
  const size_t nx = static_cast<size_t>(M) * K * esz;
  if (overlaps(workspace, need, X, nx)) return CONVROT_ERR_ALIAS;
  if (int st = check_weights(weights, n_weights, M, K, X, nx, workspace, need)) return st;
  for (int j = 0; j < n_weights; ++j) {
    const convrot_weight& w = weights[j];
    if (w.N == 0) continue;
    if (overlaps(workspace, need, w.scale, w.N * 4) || overlaps(workspace, need, w.bias, w.N * 4))
      return CONVROT_ERR_ALIAS;
  }
  if (int st = check_device()) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __half* x16 = reinterpret_cast<__half*>(ws);
  float* s_x = reinterpret_cast<float*>(ws + round256(static_cast<size_t>(M) * K * 2));
  int st = launch_pack(X, x_dtype, M, K, G, x16, kPackF16, s_x, s, input_scale);
  if (st) return st;
  return launch_grouped(x16, s_x, M, K, weights, n_weights, s, input_scale,
                        sync_at(ws + need - CONVROT_GEMM_SYNC_BYTES));
}

int convrot_pack_prologue(const float* X, int64_t M, int64_t K, int G, const convrot_prologue* pro,
                          int8_t* Q_x, float* s_x, void* stream) {
  if (!pro) return CONVROT_ERR_ARG;
  if (int st = pack_checks(X, CONVROT_F32, M, K, G, Q_x, 1, s_x)) return st;
  if (M == 0) return CONVROT_OK;
  if ((pro->weight && !aligned16(pro->weight)) || (pro->scale && !aligned16(pro->scale)) ||
      (pro->shift && !aligned16(pro->shift)))
    return CONVROT_ERR_ALIGN;
  return launch_pack_modulated(X, M, K, G, pro->weight, pro->scale, pro->shift, pro->rmsnorm != 0, pro->eps, Q_x,
                               kPackI8, s_x, static_cast<cudaStream_t>(stream));
}

int convrot_linear_prologue(const float* X, int64_t M, int64_t K, int G, const convrot_prologue* pro,
                            const convrot_weight* weights, int n_weights, void* workspace,
                            size_t workspace_bytes, void* stream) {
  if (!pro) return CONVROT_ERR_ARG;
  if (M < 0 || K <= 0) return CONVROT_ERR_ARG;
  if (int st = check_weight_list(weights, n_weights)) return st;
  if (M == 0) return CONVROT_OK;
  if (!X) return CONVROT_ERR_ARG;
  if (!valid_group(G, K)) return CONVROT_ERR_GROUP;
  if (K % 16 != 0 || !aligned16(X) || (workspace && !aligned16(workspace))) return CONVROT_ERR_ALIGN;
  if ((pro->weight && !aligned16(pro->weight)) || (pro->scale && !aligned16(pro->scale)) ||
      (pro->shift && !aligned16(pro->shift)))
    return CONVROT_ERR_ALIGN;
  if (K > CONVROT_PACK_MAX_K) return CONVROT_ERR_UNSUPPORTED;
  if (M > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
  const size_t need = convrot_linear_workspace_size(M, K);
  if (!workspace || workspace_bytes < need) return CONVROT_ERR_WORKSPACE;
  const size_t nx = static_cast<size_t>(M) * K * 4;
  if (overlaps(workspace, need, X, nx)) return CONVROT_ERR_ALIAS;
  if (int st = check_weights(weights, n_weights, M, K, X, nx, workspace, need)) return st;
  if (int st = check_device()) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __half* x16 = reinterpret_cast<__half*>(ws);
  float* s_x = reinterpret_cast<float*>(ws + round256(static_cast<size_t>(M) * K * 2));
  int st = launch_pack_modulated(X, M, K, G, pro->weight, pro->scale, pro->shift, pro->rmsnorm != 0, pro->eps, x16,
                                 kPackF16, s_x, s);
  if (st) return st;
  return launch_grouped(x16, s_x, M, K, weights, n_weights, s, 1.0f, sync_at(ws + need - CONVROT_GEMM_SYNC_BYTES));
}

int convrot_w4_expand(const uint8_t* Q_w4, int64_t N, int64_t K, int8_t* Q_w, uint16_t* Q_w16, void* stream) {
  if (N < 0 || K <= 0) return CONVROT_ERR_ARG;
  if (N == 0) return CONVROT_OK;
  if (!Q_w4 || (!Q_w && !Q_w16)) return CONVROT_ERR_ARG;
  if (K % 16 != 0 || !aligned16(Q_w4) || (Q_w && !aligned16(Q_w)) || (Q_w16 && !aligned16(Q_w16)))
    return CONVROT_ERR_ALIGN;
  if (N > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
  const size_t n = static_cast<size_t>(N) * K;
  if (overlaps(Q_w4, n / 2, Q_w, n) || overlaps(Q_w4, n / 2, Q_w16, n * 2) || overlaps(Q_w, n, Q_w16, n * 2))
    return CONVROT_ERR_ALIAS;
  if (int st = check_device()) return st;
  return launch_w4_expand(Q_w4, static_cast<int64_t>(n), Q_w, reinterpret_cast<__half*>(Q_w16),
                          static_cast<cudaStream_t>(stream));
}

int convrot_weight_chunks(const int8_t* Q_w, int64_t N, int64_t K, int32_t* kchunk, void* stream) {
  if (N < 0 || K <= 0) return CONVROT_ERR_ARG;
  if (N == 0) return CONVROT_OK;
  if (!Q_w || !kchunk) return CONVROT_ERR_ARG;
  if (K % 16 != 0 || !aligned16(Q_w) || (reinterpret_cast<uintptr_t>(kchunk) & 3u)) return CONVROT_ERR_ALIGN;
  if (K > CONVROT_MAX_K) return CONVROT_ERR_OVERFLOW;
  if (N > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
  const size_t nb = static_cast<size_t>((N + CONVROT_CHUNK_ROWS - 1) / CONVROT_CHUNK_ROWS) * 4;
  if (overlaps(Q_w, static_cast<size_t>(N) * K, kchunk, nb)) return CONVROT_ERR_ALIAS;
  if (int st = check_device()) return st;
  return launch_chunk_plan(Q_w, N, K, kchunk, static_cast<cudaStream_t>(stream));
}

int convrot_device_status(void* stream) {
  if (int st = check_device()) return st;
  const int gemm_st = read_and_clear_device_error(static_cast<cudaStream_t>(stream));
  const int w4_st = read_and_clear_w4_error();
  const int pack_st = read_and_clear_pack_error();
  return gemm_st != CONVROT_OK ? gemm_st : (w4_st != CONVROT_OK ? w4_st : pack_st);
}

size_t int8_gemm_s32_w4_workspace_size(int64_t M, int64_t K) {
  if (M < 0 || K < 0) return 0;
  return round256(static_cast<size_t>(M) * K * 2) + CONVROT_GEMM_SYNC_BYTES;
}

int int8_gemm_s32_w4(const int8_t* Q_x, int64_t M, int64_t K, const uint8_t* Q_w4, int64_t N, int32_t* A,
                     void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 0 || N < 0 || K <= 0) return CONVROT_ERR_ARG;
  if (M == 0 || N == 0) return CONVROT_OK;
  if (!Q_x || !Q_w4 || !A) return CONVROT_ERR_ARG;
  if (M > 0x7fffffff || N > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
  if (K % 64 != 0 || !aligned16(Q_x) || !aligned16(Q_w4) || !aligned16(A) || (workspace && !aligned16(workspace)))
    return CONVROT_ERR_ALIGN;
  if (K > CONVROT_W4_MAX_K) return CONVROT_ERR_UNSUPPORTED;
  const size_t need = int8_gemm_s32_w4_workspace_size(M, K);
  if (!workspace || workspace_bytes < need) return CONVROT_ERR_WORKSPACE;
  const size_t na = static_cast<size_t>(M) * N * 4, mk = static_cast<size_t>(M) * K, nk = static_cast<size_t>(N) * K / 2;
  if (overlaps(A, na, Q_x, mk) || overlaps(A, na, Q_w4, nk) || overlaps(A, na, workspace, need) ||
      overlaps(workspace, need, Q_x, mk) || overlaps(workspace, need, Q_w4, nk))
    return CONVROT_ERR_ALIAS;
  if (int st = check_device()) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __half* x16 = reinterpret_cast<__half*>(ws);
  if (int st = launch_widen(Q_x, x16, M * K, s)) return st;
  GemmLinear lin{nullptr, nullptr, nullptr, A, N, nullptr};
  lin.w4 = Q_w4;
  return launch_gemm_w4(x16, nullptr, M, K, &lin, 1, true, s, sync_at(ws + need - CONVROT_GEMM_SYNC_BYTES));
}

}  // extern "C"
