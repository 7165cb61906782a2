// mlp.cu -- convrot_mlp: an up linear, its activation, and a down linear,
// entirely on the device.
//
// X is packed once for the up linear and the up GEMM writes Y_up in fp32; the
// activation is applied as Y_up is loaded by the pack for the down linear (the
// pack's prologue), so H = act(Y_up) is never stored, and the down GEMM writes
// Y. Y_up and both packed activations live in the caller's workspace (or Y_up
// in the caller's array), so nothing goes through the host between the two
// linears.
#include "common.cuh"

namespace convrot {
namespace {

struct MlpLayout {
  size_t x16, s_x, h, h16, s_h, sync, total;
};

MlpLayout mlp_layout(int64_t M, int64_t K, int64_t N_up) {
  MlpLayout l;
  const size_t m = static_cast<size_t>(M);
  l.x16 = 0;
  l.s_x = l.x16 + round256(m * K * 2);
  l.h = l.s_x + round256(m * 4);
  l.h16 = l.h + round256(m * N_up * 4);
  l.s_h = l.h16 + round256(m * N_up * 2);
  l.sync = l.s_h + round256(m * 4);
  l.total = l.sync + CONVROT_GEMM_SYNC_BYTES;
  return l;
}

}  // namespace
}  // namespace convrot

using namespace convrot;

extern "C" size_t convrot_mlp_workspace_size(int64_t M, int64_t K, int64_t N_up) {
  if (M < 0 || K < 0 || N_up < 0) return 0;
  return mlp_layout(M, K, N_up).total;
}

extern "C" int convrot_mlp(const void* X, int x_dtype, int64_t M, int64_t K, int G_up,
                           const convrot_weight* up, int activation, int G_down,
                           const convrot_weight* down, void* workspace, size_t workspace_bytes,
                           void* stream) {
  if (M < 0 || K <= 0) return CONVROT_ERR_ARG;
  if (x_dtype != CONVROT_F32 && x_dtype != CONVROT_F16) return CONVROT_ERR_ARG;
  if (activation != CONVROT_ACT_NONE && activation != CONVROT_ACT_GELU) return CONVROT_ERR_ARG;
  if (!up || !down || up->N <= 0 || down->N <= 0 || !down->Y) return CONVROT_ERR_ARG;
  if ((!up->q16) == (!up->q4) || (!down->q16) == (!down->q4)) return CONVROT_ERR_ARG;  // one kind of weight each
  if (M == 0) return CONVROT_OK;
  if (!X) return CONVROT_ERR_ARG;
  const int64_t N_up = up->N;
  if (!valid_group(G_up, K) || !valid_group(G_down, N_up)) return CONVROT_ERR_GROUP;
  if (K % 16 != 0 || N_up % 16 != 0 || !aligned16(X) || (workspace && !aligned16(workspace)))
    return CONVROT_ERR_ALIGN;
  if (K > CONVROT_PACK_MAX_K || N_up > CONVROT_PACK_MAX_K) return CONVROT_ERR_UNSUPPORTED;
  if (M > 0x7fffffff || N_up > 0x7fffffff || down->N > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
  const MlpLayout l = mlp_layout(M, K, N_up);
  if (!workspace || workspace_bytes < l.total) return CONVROT_ERR_WORKSPACE;
  const size_t esz = x_dtype == CONVROT_F32 ? 4 : 2;
  const size_t nx = static_cast<size_t>(M) * K * esz;
  // the up linear writes H (its own Y, or the workspace); the down linear reads it
  convrot_weight up_w = *up;
  float* H = up->Y ? up->Y : reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + l.h);
  up_w.Y = H;
  if (overlaps(workspace, l.total, X, nx)) return CONVROT_ERR_ALIAS;
  if (int st = check_weights(&up_w, 1, M, K, X, nx, up->Y ? workspace : nullptr, up->Y ? l.total : 0)) return st;
  const size_t nh = static_cast<size_t>(M) * N_up * 4;
  if (int st = check_weights(down, 1, M, N_up, H, nh, workspace, l.total)) return st;
  if (overlaps(down->Y, static_cast<size_t>(M) * down->N * 4, X, nx)) return CONVROT_ERR_ALIAS;
  if (int st = check_device()) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __half* x16 = reinterpret_cast<__half*>(ws + l.x16);
  float* s_x = reinterpret_cast<float*>(ws + l.s_x);
  __half* h16 = reinterpret_cast<__half*>(ws + l.h16);
  float* s_h = reinterpret_cast<float*>(ws + l.s_h);
  if (int st = launch_pack(X, x_dtype, M, K, G_up, x16, kPackF16, s_x, s)) return st;
  const GemmLinear lu = to_linear(*up, H);
  const GemmSync sync = sync_at(ws + l.sync);  // the two GEMMs run one after the other
  if (int st = launch_linears(x16, s_x, M, K, &lu, 1, false, s, sync)) return st;
  int st = (activation == CONVROT_ACT_GELU) ? launch_pack_gelu(H, M, N_up, G_down, h16, s_h, s)
                                             : launch_pack(H, CONVROT_F32, M, N_up, G_down, h16, kPackF16, s_h, s);
  if (st) return st;
  const GemmLinear ld = to_linear(*down, down->Y);
  return launch_linears(h16, s_h, M, N_up, &ld, 1, false, s, sync);
}
