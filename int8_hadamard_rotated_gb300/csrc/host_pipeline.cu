// host_pipeline.cu -- convrot_linear_host: the fused convrot linear with its
// activation input and outputs in host memory.
//
// The rows are processed in chunks. Every chunk is copied in on the caller's
// copy-in stream, packed and multiplied (one grouped GEMM over all linears)
// on the compute stream, and its output rows copied back on the copy-out
// stream, with events ordering the three: the transfers of one chunk overlap
// the compute and transfers of its neighbours. Device buffers (input rows,
// packed activation, output rows) are double-buffered in the caller's
// workspace; a buffer is refilled only after the work that read it finished.
#include "common.cuh"

#include <cstring>

namespace convrot {
namespace {

struct ChunkBuffers {
  uint8_t* x;      // [chunk_rows, K] input rows (x dtype)
  __half* q16;     // [chunk_rows, K] binary16 codes
  float* s_x;      // [chunk_rows] row scales
  float* y;        // output rows of every linear, back to back: [chunk_rows, N_j] each
};

size_t esize(int x_dtype) { return x_dtype == CONVROT_F32 ? 4 : 2; }

// Bytes of one of the two buffer sets.
size_t buffer_set_bytes(int64_t chunk_rows, int64_t K, int x_dtype, int64_t n_total) {
  const size_t r = static_cast<size_t>(chunk_rows);
  return round256(r * K * esize(x_dtype)) + round256(r * K * 2) + round256(r * 4) + round256(r * n_total * 4);
}

ChunkBuffers carve(uint8_t* base, int64_t chunk_rows, int64_t K, int x_dtype) {
  const size_t r = static_cast<size_t>(chunk_rows);
  ChunkBuffers b;
  b.x = base;
  b.q16 = reinterpret_cast<__half*>(base + round256(r * K * esize(x_dtype)));
  b.s_x = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(b.q16) + round256(r * K * 2));
  b.y = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(b.s_x) + round256(r * 4));
  return b;
}

constexpr int64_t kDefaultChunkRows = 768;
constexpr int64_t kFirstChunkRows = 256;  // the default's first chunk

int64_t chunk_rows_for(int64_t M, int64_t chunk_rows) {
  const int64_t c = chunk_rows > 0 ? chunk_rows : kDefaultChunkRows;
  return c < M ? c : M;
}

// Rows of chunk c. With the default chunk size the first chunk is shorter:
// its copy-in and compute are the pipeline's fill before the first copy-out
// (measured on the DiT projections: 256 then 768 rows 1.05 ms; 768 rows
// throughout 1.08 ms; 256, 512, then 768 rows 1.07 ms). With an explicit
// chunk size, that size.
int64_t chunk_rows_at(int64_t c, int64_t cr, int64_t chunk_rows) {
  if (chunk_rows > 0 || c > 0) return cr;
  return kFirstChunkRows < cr ? kFirstChunkRows : cr;
}

struct Events {
  cudaEvent_t start = nullptr;
  cudaEvent_t in[2] = {nullptr, nullptr};    // input rows landed
  cudaEvent_t packed[2] = {nullptr, nullptr};  // input buffer read by the pack
  cudaEvent_t done[2] = {nullptr, nullptr};  // outputs written
  cudaEvent_t out[2] = {nullptr, nullptr};   // outputs copied back
  ~Events() {
    // destroying an event that is still pending is allowed; it is released when it completes
    cudaEvent_t* all[] = {&start, &in[0], &in[1], &packed[0], &packed[1], &done[0], &done[1], &out[0], &out[1]};
    for (cudaEvent_t* e : all)
      if (*e) cudaEventDestroy(*e);
  }
  int create() {
    cudaEvent_t* all[] = {&start, &in[0], &in[1], &packed[0], &packed[1], &done[0], &done[1], &out[0], &out[1]};
    for (cudaEvent_t* e : all) {
      cudaError_t err = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
      if (err != cudaSuccess) return set_cuda_error(err);
    }
    return CONVROT_OK;
  }
};

#define CONVROT_TRY(call)                                  \
  do {                                                     \
    cudaError_t err_ = (call);                             \
    if (err_ != cudaSuccess) return set_cuda_error(err_);  \
  } while (0)

}  // namespace
}  // namespace convrot

using namespace convrot;

extern "C" size_t convrot_linear_host_workspace_size(int64_t M, int64_t K, int x_dtype, int64_t n_total,
                                                     int64_t chunk_rows) {
  if (M <= 0 || K <= 0 || n_total < 0 || chunk_rows < 0) return 0;
  if (x_dtype != CONVROT_F32 && x_dtype != CONVROT_F16) return 0;
  return 2 * buffer_set_bytes(chunk_rows_for(M, chunk_rows), K, x_dtype, n_total) + CONVROT_GEMM_SYNC_BYTES;
}

extern "C" int convrot_linear_host(const void* X_host, int x_dtype, int64_t M, int64_t K, int G,
                                   const convrot_weight* weights, int n_weights, int64_t chunk_rows,
                                   void* workspace, size_t workspace_bytes, void* stream,
                                   void* copy_in_stream, void* copy_out_stream) {
  if (M < 0 || K <= 0 || chunk_rows < 0) return CONVROT_ERR_ARG;
  if (x_dtype != CONVROT_F32 && x_dtype != CONVROT_F16) return CONVROT_ERR_ARG;
  if (int st = check_weight_list(weights, n_weights)) return st;
  if (M == 0) return CONVROT_OK;
  if (!X_host) return CONVROT_ERR_ARG;
  if (!valid_group(G, K)) return CONVROT_ERR_GROUP;
  if (K % 16 != 0 || (workspace && !aligned16(workspace))) return CONVROT_ERR_ALIGN;
  if (K > CONVROT_PACK_MAX_K) return CONVROT_ERR_UNSUPPORTED;
  if (M > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
  int64_t n_total = 0;
  for (int j = 0; j < n_weights; ++j) n_total += weights[j].N;
  const size_t need = convrot_linear_host_workspace_size(M, K, x_dtype, n_total, chunk_rows);
  if (!workspace || workspace_bytes < need) return CONVROT_ERR_WORKSPACE;
  for (int j = 0; j < n_weights; ++j) {
    const convrot_weight& w = weights[j];
    if (w.N == 0) continue;
    if (!aligned16(weight_codes(w)) || (w.scale && !aligned16(w.scale)) || (w.bias && !aligned16(w.bias)))
      return CONVROT_ERR_ALIGN;
    if (w.q4) {
      if (K % 64 != 0 || w.N % 4 != 0) return CONVROT_ERR_ALIGN;
      if (K > CONVROT_W4_MAX_K) return CONVROT_ERR_UNSUPPORTED;
    }
    if (overlaps(workspace, need, weight_codes(w), weight_code_bytes(w, K)) ||
        overlaps(workspace, need, w.scale, static_cast<size_t>(w.N) * 4) ||
        overlaps(workspace, need, w.bias, static_cast<size_t>(w.N) * 4))
      return CONVROT_ERR_ALIAS;
  }
  if (int st = check_device()) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStream_t sin = copy_in_stream ? static_cast<cudaStream_t>(copy_in_stream) : s;
  cudaStream_t sout = copy_out_stream ? static_cast<cudaStream_t>(copy_out_stream) : s;
  Events ev;
  if (int st = ev.create()) return st;
  CONVROT_TRY(cudaEventRecord(ev.start, s));
  CONVROT_TRY(cudaStreamWaitEvent(sin, ev.start, 0));
  CONVROT_TRY(cudaStreamWaitEvent(sout, ev.start, 0));

  const int64_t cr = chunk_rows_for(M, chunk_rows);
  const size_t set_bytes = buffer_set_bytes(cr, K, x_dtype, n_total);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const ChunkBuffers B[2] = {carve(ws, cr, K, x_dtype), carve(ws + set_bytes, cr, K, x_dtype)};
  const GemmSync sync = sync_at(ws + 2 * set_bytes);  // the chunks' GEMMs run one after the other on `stream`
  const size_t esz = esize(x_dtype);
  const uint8_t* xh = static_cast<const uint8_t*>(X_host);
  int64_t r0 = 0;
  int64_t nchunks = 0;
  for (int64_t c = 0; r0 < M; ++c, ++nchunks) {
    const int b = static_cast<int>(c & 1);
    const int64_t rows = chunk_rows_at(c, cr, chunk_rows);
    const int64_t m = (M - r0) < rows ? (M - r0) : rows;
    // copy in, once the pack two chunks back has read this input buffer
    if (c >= 2) CONVROT_TRY(cudaStreamWaitEvent(sin, ev.packed[b], 0));
    CONVROT_TRY(cudaMemcpyAsync(B[b].x, xh + static_cast<size_t>(r0) * K * esz, static_cast<size_t>(m) * K * esz,
                                cudaMemcpyHostToDevice, sin));
    CONVROT_TRY(cudaEventRecord(ev.in[b], sin));
    // pack and multiply, once the copy-out two chunks back has read this output buffer
    CONVROT_TRY(cudaStreamWaitEvent(s, ev.in[b], 0));
    if (c >= 2) CONVROT_TRY(cudaStreamWaitEvent(s, ev.out[b], 0));
    if (int st = launch_pack(B[b].x, x_dtype, m, K, G, B[b].q16, kPackF16, B[b].s_x, s)) return st;
    CONVROT_TRY(cudaEventRecord(ev.packed[b], s));
    GemmLinear lins[CONVROT_MAX_LINEARS];
    int n = 0;
    size_t off = 0;
    for (int j = 0; j < n_weights; ++j) {
      const convrot_weight& w = weights[j];
      if (w.N == 0) continue;
      lins[n++] = to_linear(w, B[b].y + off);
      off += static_cast<size_t>(m) * w.N;
    }
    if (n > 0)
      if (int st = launch_linears(B[b].q16, B[b].s_x, m, K, lins, n, false, s, sync)) return st;
    CONVROT_TRY(cudaEventRecord(ev.done[b], s));
    // copy out every linear's rows of this chunk (contiguous in both places)
    CONVROT_TRY(cudaStreamWaitEvent(sout, ev.done[b], 0));
    off = 0;
    for (int j = 0; j < n_weights; ++j) {
      const convrot_weight& w = weights[j];
      if (w.N == 0) continue;
      const size_t bytes = static_cast<size_t>(m) * w.N * 4;
      CONVROT_TRY(cudaMemcpyAsync(w.Y + static_cast<size_t>(r0) * w.N, B[b].y + off, bytes,
                                  cudaMemcpyDeviceToHost, sout));
      off += static_cast<size_t>(m) * w.N;
    }
    CONVROT_TRY(cudaEventRecord(ev.out[b], sout));
    r0 += m;
  }
  // later work on `stream` follows every copy-out
  CONVROT_TRY(cudaStreamWaitEvent(s, ev.out[0], 0));
  if (nchunks > 1) CONVROT_TRY(cudaStreamWaitEvent(s, ev.out[1], 0));
  return CONVROT_OK;
}

// ---------------------------------------------------------------------------
// convrot_mlp_host: the MLP pair with X and Y in host memory, pipelined the
// same way. Per chunk: input rows and output rows in double-buffered chunk
// buffers, and one convrot_mlp workspace, reused by every chunk since the
// chunks' calls follow one another on the compute stream.
// ---------------------------------------------------------------------------

namespace convrot {
namespace {

constexpr int64_t kMlpChunkRows = 1536;  // 3 chunks of the DiT MLP's 4608 rows measured fastest

int64_t mlp_chunk_rows_for(int64_t M, int64_t chunk_rows) {
  const int64_t c = chunk_rows > 0 ? chunk_rows : kMlpChunkRows;
  return c < M ? c : M;
}

size_t mlp_set_bytes(int64_t cr, int64_t K, int x_dtype, int64_t N_down) {
  const size_t r = static_cast<size_t>(cr);
  return round256(r * K * esize(x_dtype)) + round256(r * N_down * 4);
}

}  // namespace
}  // namespace convrot

extern "C" size_t convrot_mlp_host_workspace_size(int64_t M, int64_t K, int x_dtype, int64_t N_up,
                                                  int64_t N_down, int64_t chunk_rows) {
  if (M <= 0 || K <= 0 || N_up <= 0 || N_down <= 0 || chunk_rows < 0) return 0;
  if (x_dtype != CONVROT_F32 && x_dtype != CONVROT_F16) return 0;
  const int64_t cr = mlp_chunk_rows_for(M, chunk_rows);
  return 2 * mlp_set_bytes(cr, K, x_dtype, N_down) + round256(convrot_mlp_workspace_size(cr, K, N_up));
}

extern "C" int convrot_mlp_host(const void* X_host, int x_dtype, int64_t M, int64_t K, int G_up,
                                const convrot_weight* up, int activation, int G_down,
                                const convrot_weight* down, float* Y_host, int64_t chunk_rows,
                                void* workspace, size_t workspace_bytes, void* stream,
                                void* copy_in_stream, void* copy_out_stream) {
  if (M < 0 || K <= 0 || chunk_rows < 0 || !up || !down) return CONVROT_ERR_ARG;
  if (x_dtype != CONVROT_F32 && x_dtype != CONVROT_F16) return CONVROT_ERR_ARG;
  if (activation != CONVROT_ACT_NONE && activation != CONVROT_ACT_GELU && activation != CONVROT_ACT_SWIGLU)
    return CONVROT_ERR_ARG;
  const int n_up = activation == CONVROT_ACT_SWIGLU ? 2 : 1;
  const int64_t N_up = up[0].N, N_down = down->N;
  if (N_up <= 0 || N_down <= 0) return CONVROT_ERR_ARG;
  if (M == 0) return CONVROT_OK;
  if (!X_host || !Y_host) return CONVROT_ERR_ARG;
  if (workspace && !aligned16(workspace)) return CONVROT_ERR_ALIGN;
  if (M > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
  const size_t need = convrot_mlp_host_workspace_size(M, K, x_dtype, N_up, N_down, chunk_rows);
  if (need == 0) return CONVROT_ERR_ARG;
  if (!workspace || workspace_bytes < need) return CONVROT_ERR_WORKSPACE;
  if (int st = check_device()) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStream_t sin = copy_in_stream ? static_cast<cudaStream_t>(copy_in_stream) : s;
  cudaStream_t sout = copy_out_stream ? static_cast<cudaStream_t>(copy_out_stream) : s;
  Events ev;
  if (int st = ev.create()) return st;
  CONVROT_TRY(cudaEventRecord(ev.start, s));
  CONVROT_TRY(cudaStreamWaitEvent(sin, ev.start, 0));
  CONVROT_TRY(cudaStreamWaitEvent(sout, ev.start, 0));

  const int64_t cr = mlp_chunk_rows_for(M, chunk_rows);
  const size_t set_bytes = mlp_set_bytes(cr, K, x_dtype, N_down);
  const size_t esz = esize(x_dtype);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* xbuf[2] = {ws, ws + set_bytes};
  float* ybuf[2] = {reinterpret_cast<float*>(ws + round256(static_cast<size_t>(cr) * K * esz)),
                    reinterpret_cast<float*>(ws + set_bytes + round256(static_cast<size_t>(cr) * K * esz))};
  uint8_t* mlp_ws = ws + 2 * set_bytes;
  const size_t mlp_ws_bytes = workspace_bytes - 2 * set_bytes;
  // the descriptors with the chunk buffers as outputs (H stays in the MLP workspace)
  convrot_weight up_c[2], down_c = *down;
  for (int j = 0; j < n_up; ++j) {
    up_c[j] = up[j];
    up_c[j].Y = nullptr;
  }
  const uint8_t* xh = static_cast<const uint8_t*>(X_host);
  int64_t r0 = 0, nchunks = 0;
  for (int64_t c = 0; r0 < M; ++c, ++nchunks) {
    const int b = static_cast<int>(c & 1);
    const int64_t m = (M - r0) < cr ? (M - r0) : cr;
    // copy in, once the call two chunks back has finished with this input buffer
    if (c >= 2) CONVROT_TRY(cudaStreamWaitEvent(sin, ev.done[b], 0));
    CONVROT_TRY(cudaMemcpyAsync(xbuf[b], xh + static_cast<size_t>(r0) * K * esz, static_cast<size_t>(m) * K * esz,
                                cudaMemcpyHostToDevice, sin));
    CONVROT_TRY(cudaEventRecord(ev.in[b], sin));
    // the pair on the chunk, once the copy-out two chunks back has read this output buffer
    CONVROT_TRY(cudaStreamWaitEvent(s, ev.in[b], 0));
    if (c >= 2) CONVROT_TRY(cudaStreamWaitEvent(s, ev.out[b], 0));
    down_c.Y = ybuf[b];
    if (int st = convrot_mlp(xbuf[b], x_dtype, m, K, G_up, up_c, activation, G_down, &down_c, mlp_ws, mlp_ws_bytes,
                             s))
      return st;
    CONVROT_TRY(cudaEventRecord(ev.done[b], s));
    // copy out the chunk's rows of Y
    CONVROT_TRY(cudaStreamWaitEvent(sout, ev.done[b], 0));
    CONVROT_TRY(cudaMemcpyAsync(Y_host + static_cast<size_t>(r0) * N_down, ybuf[b],
                                static_cast<size_t>(m) * N_down * 4, cudaMemcpyDeviceToHost, sout));
    CONVROT_TRY(cudaEventRecord(ev.out[b], sout));
    r0 += m;
  }
  // later work on `stream` follows every copy-out
  CONVROT_TRY(cudaStreamWaitEvent(s, ev.out[0], 0));
  if (nchunks > 1) CONVROT_TRY(cudaStreamWaitEvent(s, ev.out[1], 0));
  return CONVROT_OK;
}
