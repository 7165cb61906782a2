// mlp.cu -- convrot_mlp: an up linear, its activation, and a down linear,
// entirely on the device.
//
// X is packed once for the up GEMM, which applies the activation to its
// output in its epilogue and writes only H = act(Y_up) in fp32: GELU
// elementwise, or split SwiGLU h = silu(gate) * up of a gate and an up
// weight sharing the input ("ggml operator extensions", sd.cpp integration:
// the GEMM epilogue writes only the activated output). H is then packed for
// the down linear and the down GEMM writes Y. H and both packed activations
// live in the caller's workspace (or H in the caller's array), so nothing
// goes through the host between the two linears.
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
  if (activation != CONVROT_ACT_NONE && activation != CONVROT_ACT_GELU && activation != CONVROT_ACT_SWIGLU)
    return CONVROT_ERR_ARG;
  const int n_up = (activation == CONVROT_ACT_SWIGLU) ? 2 : 1;  // gate and up, or the up linear
  if (!up || !down || down->N <= 0 || !down->Y) return CONVROT_ERR_ARG;
  for (int j = 0; j < n_up; ++j)
    if (up[j].N <= 0 || (!up[j].q16) == (!up[j].q4)) return CONVROT_ERR_ARG;  // one kind of weight each
  if ((!down->q16) == (!down->q4)) return CONVROT_ERR_ARG;
  if (n_up == 2 && up[1].N != up[0].N) return CONVROT_ERR_ARG;
  if (n_up == 2 && (!up[0].q16 || !up[1].q16)) return CONVROT_ERR_UNSUPPORTED;  // split SwiGLU: binary16 weights
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
  // the up GEMM writes H (the caller's array up[0].Y, or the workspace); the down linear reads it
  convrot_weight up_w[2] = {up[0], n_up == 2 ? up[1] : up[0]};
  float* H = up->Y ? up->Y : reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + l.h);
  for (int j = 0; j < n_up; ++j) up_w[j].Y = H;
  if (overlaps(workspace, l.total, X, nx)) return CONVROT_ERR_ALIAS;
  // the gate and up linears share H as their output: check each against the inputs alone
  for (int j = 0; j < n_up; ++j)
    if (int st = check_weights(&up_w[j], 1, M, K, X, nx, up->Y ? workspace : nullptr, up->Y ? l.total : 0))
      return st;
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
  const GemmLinear lu[2] = {to_linear(up_w[0], H), to_linear(up_w[1], H)};
  const GemmSync sync = sync_at(ws + l.sync);  // the two GEMMs run one after the other
  // the activation in the up GEMM's epilogue (GELU on fp32 pairs costs the
  // GEMM about 4 %; applied in the repack instead it costs that kernel about
  // 35 %), then the plain repack of H
  if (int st = launch_gemm_act(x16, s_x, M, K, lu, n_up, activation, s, sync)) return st;
  if (int st = launch_pack(H, CONVROT_F32, M, N_up, G_down, h16, kPackF16, s_h, s)) return st;
  const GemmLinear ld = to_linear(*down, down->Y);
  return launch_linears(h16, s_h, M, N_up, &ld, 1, false, s, sync);
}

extern "C" int convrot_linear_swiglu(const void* X, int x_dtype, int64_t M, int64_t K, int G,
                                     const convrot_weight* gate_up, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  if (M < 0 || K <= 0) return CONVROT_ERR_ARG;
  if (x_dtype != CONVROT_F32 && x_dtype != CONVROT_F16) return CONVROT_ERR_ARG;
  if (!gate_up || gate_up[0].N <= 0 || gate_up[1].N != gate_up[0].N || !gate_up[0].Y) return CONVROT_ERR_ARG;
  if (!gate_up[0].q16 || !gate_up[1].q16) return CONVROT_ERR_ARG;  // binary16 weights
  if (gate_up[0].q4 || gate_up[1].q4) return CONVROT_ERR_ARG;
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
  convrot_weight w[2] = {gate_up[0], gate_up[1]};
  w[1].Y = w[0].Y;  // one output: h
  for (int j = 0; j < 2; ++j) {
    if (int st = check_weights(&w[j], 1, M, K, X, nx, workspace, need)) return st;
    if (overlaps(workspace, need, w[j].scale, w[j].N * 4) || overlaps(workspace, need, w[j].bias, w[j].N * 4))
      return CONVROT_ERR_ALIAS;
  }
  // h must not overlap the other weight's arrays either
  const size_t ny = static_cast<size_t>(M) * w[0].N * 4;
  for (int j = 0; j < 2; ++j)
    if (overlaps(w[0].Y, ny, w[j].q16, static_cast<size_t>(w[j].N) * K * 2) ||
        overlaps(w[0].Y, ny, w[j].scale, w[j].N * 4) || overlaps(w[0].Y, ny, w[j].bias, w[j].N * 4))
      return CONVROT_ERR_ALIAS;
  if (int st = check_device()) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __half* x16 = reinterpret_cast<__half*>(ws);
  float* s_x = reinterpret_cast<float*>(ws + round256(static_cast<size_t>(M) * K * 2));
  if (int st = launch_pack(X, x_dtype, M, K, G, x16, kPackF16, s_x, s)) return st;
  const GemmLinear lins[2] = {to_linear(w[0], w[0].Y), to_linear(w[1], w[0].Y)};
  return launch_gemm_act(x16, s_x, M, K, lins, 2, CONVROT_ACT_SWIGLU, s, sync_at(ws + need - CONVROT_GEMM_SYNC_BYTES));
}
