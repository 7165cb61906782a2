// gemm.cu -- the exact INT8 x INT8 -> INT32 GEMM with the fused convrot
// reconstruction, on the sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// What it computes (stable-diffusion.cpp docs, page "INT8 Convrot
// Safetensors", "Runtime activation quantization"): A[r,o] = sum_i
// Q_x[r,i] Q_w[o,i] accumulated in signed 32-bit integers, then
// Y[r,o] = float(A[r,o]) * s_x[r] * s_w[o] + b[o], evaluated in that order
// with one fp32 rounding per operation (page "ggml operator extensions",
// "sd.cpp integration"); the weight scale and bias are optional.
//
// Exactness on fp16 tensor cores. sm_103a has no 8-bit integer MMA kind, so
// both operands are the int8 codes stored as binary16 (every integer in
// [-127, 127] is exact). Each product is an integer of magnitude <= 127^2,
// and a run of at most 1024 of them keeps every partial sum below
// 1024 * 127^2 = 16,516,096 < 2^24, where fp32 represents every integer: the
// fp32 tensor-memory accumulator of one 1024-deep K-chunk therefore holds the
// exact integer. The epilogue warps convert each finished chunk to int32 and
// add it into per-thread int32 registers, so A is bit-exact for any K up to
// the int32 limit.
//
// Kernel shape. One persistent CTA per SM, 10 warps:
//   warps 0-7  epilogue: drain TMEM chunks into int32 registers, reconstruct,
//              store (each thread owns one output feature o and 128
//              activation rows of a tile; a warp stores 128 B per row).
//   warp 8     TMA producer: streams 128x64 weight and 256x64 activation
//              fp16 tiles (128-byte swizzle) into a 4-stage ring.
//   warp 9     MMA issuer: one thread issues tcgen05.mma kind::f16,
//              M=128 (weight rows) x N=256 (activation rows) x K=16, into one
//              of two 256-column fp32 TMEM buffers that alternate per chunk,
//              so the epilogue drains one while the other accumulates.
// Tiles of all linears sharing the input are enumerated activation-tile-major
// (every weight tile of every linear for one 256-row activation band, then
// the next band), so the band stays in L2 while the weights stream past it.
#include "common.cuh"

#include <cuda.h>
#include <mutex>

namespace convrot {

// Sticky device error word of the GEMM kernel (timeouts of bounded waits).
__device__ int g_device_error = 0;

namespace {

constexpr int BM = 128;               // weight rows per tile (MMA M)
constexpr int BN = 256;               // activation rows per tile (MMA N)
constexpr int BK = 64;                // K per pipeline stage: 64 fp16 = 128 B
constexpr int STAGES = 4;
constexpr int KB_PER_CHUNK = 16;      // 16 x 64 = 1024 products per exact chunk
constexpr int UMMA_K = 16;            // K of one kind::f16 MMA
constexpr int W_TILE_BYTES = BM * BK * 2;
constexpr int X_TILE_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = W_TILE_BYTES + X_TILE_BYTES;
constexpr int NUM_EPI_WARPS = 8;
constexpr int PRODUCER_WARP = NUM_EPI_WARPS;
constexpr int MMA_WARP = NUM_EPI_WARPS + 1;
constexpr int THREADS = (NUM_EPI_WARPS + 2) * 32;
constexpr int TMEM_COLS = 2 * BN;     // two fp32 accumulators of BN columns
constexpr int MAX_LIN = CONVROT_MAX_LINEARS;
constexpr int COLS_PER_THREAD = BN / 2;   // two epilogue warpgroups split the columns
constexpr uint32_t IDESC = idesc_f16_f32(BM, BN);
constexpr int RASTER_BANDS = 8;       // activation bands per raster group

static_assert(TMEM_COLS <= 512, "TMEM has 512 columns");
static_assert(KB_PER_CHUNK * BK * 127 * 127 < (1 << 24), "chunk must stay exact in fp32");

// shared-memory layout (after aligning the base to 1024 B)
constexpr int SMEM_STAGES = STAGES * STAGE_BYTES;
constexpr int SMEM_BARS = SMEM_STAGES;                         // full[S], empty[S], tfull[2], tempty[2], drain
constexpr int NUM_BARS = 2 * STAGES + 2 + 2 + 1;
constexpr int SMEM_MISC = SMEM_BARS + NUM_BARS * 8;            // tmem base (u32), abort flag (int)
constexpr int SMEM_TOTAL = SMEM_MISC + 16;
constexpr int SMEM_ALLOC = SMEM_TOTAL + 1024;                  // slack for the 1024-B alignment

struct GemmParams {
  CUtensorMap tmap_x;              // activation codes, fp16 [M, K]
  CUtensorMap tmap_w[MAX_LIN];     // weight codes, fp16 [N_j, K]
  const float* s_w[MAX_LIN];
  const float* bias[MAX_LIN];
  void* out[MAX_LIN];              // fp32 Y_j or int32 A_j, [M, N_j]
  int N[MAX_LIN];
  int wtile_start[MAX_LIN + 1];    // prefix sums of weight tiles per linear
  const float* s_x;
  int M;
  int K;
  int num_kb;                      // ceil(K / BK)
  int n_xtiles;                    // ceil(M / BN)
  int n_wtiles;                    // sum over linears of ceil(N_j / BM)
  int total_tiles;
  int n_lin;
  int raw_s32;
};

struct TileCoord {
  int lin, wt, xt;
};

// Raster order: tiles are taken in groups of RASTER_BANDS activation bands;
// inside a group, consecutive tiles walk the bands of one weight tile before
// moving to the next weight tile (of the same or the next linear). The ~152
// tiles in flight then cover ~RASTER_BANDS bands x ~152/RASTER_BANDS weight
// tiles, which stay in L2 while the group is swept.
__device__ __forceinline__ TileCoord decode_tile(const GemmParams& p, int t) {
  const int per_group = RASTER_BANDS * p.n_wtiles;
  const int g = t / per_group;
  const int idx = t - g * per_group;
  const int gm = min(RASTER_BANDS, p.n_xtiles - g * RASTER_BANDS);
  const int w = idx / gm;
  TileCoord c;
  c.xt = g * RASTER_BANDS + (idx - w * gm);
  int j = 0;
#pragma unroll 1
  while (j + 1 < p.n_lin && w >= p.wtile_start[j + 1]) ++j;
  c.lin = j;
  c.wt = w - p.wtile_start[j];
  return c;
}

__global__ void __launch_bounds__(THREADS, 1)
convrot_gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SMEM_BARS);
  uint64_t* full = bars;                   // [STAGES]
  uint64_t* empty = bars + STAGES;         // [STAGES]
  uint64_t* tfull = bars + 2 * STAGES;     // [2]
  uint64_t* tempty = bars + 2 * STAGES + 2;
  uint64_t* drain = bars + 2 * STAGES + 4;
  uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(smem + SMEM_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SMEM_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int* err = &g_device_error;

  if (threadIdx.x == PRODUCER_WARP * 32) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], NUM_EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&p.tmap_x);
    for (int j = 0; j < p.n_lin; ++j) tma_prefetch_desc(&p.tmap_w[j]);
  }
  if (warp == MMA_WARP) {
    tmem_alloc(tmem_base_smem, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_smem;

  const int num_chunks = (p.num_kb + KB_PER_CHUNK - 1) / KB_PER_CHUNK;

  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      const uint64_t pol_x = l2_policy_evict_normal();
      const uint64_t pol_w = l2_policy_evict_normal();
      uint32_t stage = 0, phase = 0;
      uint32_t n_issued = 0;  // stage loads issued so far (stage = n % STAGES)
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.total_tiles; t += gridDim.x) {
        const TileCoord c = decode_tile(p, t);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
          uint8_t* sw = smem + stage * STAGE_BYTES;
          uint8_t* sx = sw + W_TILE_BYTES;
          tma_load_2d(sw, &p.tmap_w[c.lin], &full[stage], kb * BK, c.wt * BM, pol_w);
          tma_load_2d(sx, &p.tmap_x, &full[stage], kb * BK, c.xt * BN, pol_x);
          ++n_issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // No copy may land after the CTA exits: wait (bounded) for the last
      // phase of every stage that was ever filled.
      for (uint32_t s = 0; s < STAGES; ++s)
        if (n_issued > s) {
          const uint32_t uses = (n_issued - 1 - s) / STAGES + 1;  // times stage s was filled
          mbar_wait(&full[s], (uses - 1) & 1u, nullptr, err);
        }
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, chunk_iter = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.total_tiles; t += gridDim.x) {
        for (int ch = 0; ok && ch < num_chunks; ++ch) {
          const uint32_t buf = chunk_iter & 1u;
          const uint32_t use = chunk_iter >> 1;
          if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort_flag, err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * BN;
          const int kb0 = ch * KB_PER_CHUNK;
          const int kb1 = min(kb0 + KB_PER_CHUNK, p.num_kb);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(&full[stage], phase, abort_flag, err)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sw = smem_u32(smem + stage * STAGE_BYTES);
            const uint64_t a_desc = smem_desc_sw128(sw);
            const uint64_t b_desc = smem_desc_sw128(sw + W_TILE_BYTES);
#pragma unroll
            for (int k = 0; k < BK / UMMA_K; ++k) {
              // advance the start address by k * 32 bytes inside the swizzle row
              const uint64_t koff = static_cast<uint64_t>((k * UMMA_K * 2) >> 4);
              mma_f16_ss(d_tmem, a_desc + koff, b_desc + koff, IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
            }
            mma_commit(&empty[stage]);
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          mma_commit(&tfull[buf]);
          ++chunk_iter;
        }
      }
      // all issued MMAs complete before TMEM is released
      mma_commit(drain);
      mbar_wait(drain, 0, nullptr, err);
    }
    __syncwarp();
  } else {
    // ------------------------------ epilogue ------------------------------
    const uint64_t pol_y = l2_policy_evict_first();
    const int quarter = warp & 3;             // TMEM lanes 32*quarter .. +31
    const int half = warp >> 2;               // activation columns half*128 .. +127
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    uint32_t chunk_iter = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < p.total_tiles; t += gridDim.x) {
      const TileCoord c = decode_tile(p, t);
      int acc[COLS_PER_THREAD];
#pragma unroll
      for (int i = 0; i < COLS_PER_THREAD; ++i) acc[i] = 0;
      for (int ch = 0; ch < num_chunks; ++ch) {
        const uint32_t buf = chunk_iter & 1u;
        const uint32_t use = chunk_iter >> 1;
        if (!mbar_wait(&tfull[buf], use & 1u, abort_flag, err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < COLS_PER_THREAD / 32; ++q) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tmem_base + lane_base + buf * BN + half * COLS_PER_THREAD + q * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[q * 32 + i] += __float2int_rz(__uint_as_float(r[i]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        ++chunk_iter;
      }
      if (!ok) break;
      const int N = p.N[c.lin];
      const int o = c.wt * BM + 32 * quarter + lane;
      const int r0 = c.xt * BN + half * COLS_PER_THREAD;
      if (o < N) {
        if (p.raw_s32) {
          int32_t* A = static_cast<int32_t*>(p.out[c.lin]);
#pragma unroll
          for (int i = 0; i < COLS_PER_THREAD; ++i) {
            const int r = r0 + i;
            if (r < p.M) st_global_hint(A + static_cast<int64_t>(r) * N + o, acc[i], pol_y);
          }
        } else {
          float* Y = static_cast<float*>(p.out[c.lin]);
          const float* sw_ptr = p.s_w[c.lin];
          const float* b_ptr = p.bias[c.lin];
          const float sw = sw_ptr ? __ldg(sw_ptr + o) : 1.0f;
          const float bb = b_ptr ? __ldg(b_ptr + o) : 0.0f;
#pragma unroll
          for (int i = 0; i < COLS_PER_THREAD; ++i) {
            const int r = r0 + i;
            if (r < p.M) {
              // float(A) * s_x * s_w + b, one rounding per operation, in that order
              float y = __fmul_rn(__int2float_rn(acc[i]), __ldg(p.s_x + r));
              if (sw_ptr) y = __fmul_rn(y, sw);
              if (b_ptr) y = __fadd_rn(y, bb);
              st_global_hint(Y + static_cast<int64_t>(r) * N + o, y, pol_y);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// fp16 [rows, K] row-major, box = box_rows x 64, 128-byte swizzle, zero fill.
int make_tmap(CUtensorMap* m, const void* base, int64_t rows, int64_t K, int box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return set_cuda_error(cudaErrorNotSupported);
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_cuda_error(cudaErrorInvalidValue);
  return CONVROT_OK;
}

}  // namespace

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

int launch_gemm(const __half* x16, const float* s_x, int64_t M, int64_t K,
                const GemmLinear* lins, int n_lin, bool raw_s32, cudaStream_t stream) {
  if (M == 0) return CONVROT_OK;
  GemmParams p;
  memset(&p, 0, sizeof(p));
  int st = make_tmap(&p.tmap_x, x16, M, K, BN);
  if (st) return st;
  int wt = 0;
  for (int j = 0; j < n_lin; ++j) {
    st = make_tmap(&p.tmap_w[j], lins[j].w16, lins[j].N, K, BM);
    if (st) return st;
    p.s_w[j] = lins[j].s_w;
    p.bias[j] = lins[j].bias;
    p.out[j] = lins[j].out;
    p.N[j] = static_cast<int>(lins[j].N);
    p.wtile_start[j] = wt;
    wt += static_cast<int>((lins[j].N + BM - 1) / BM);
  }
  p.wtile_start[n_lin] = wt;
  p.s_x = s_x;
  p.M = static_cast<int>(M);
  p.K = static_cast<int>(K);
  p.num_kb = static_cast<int>((K + BK - 1) / BK);
  p.n_xtiles = static_cast<int>((M + BN - 1) / BN);
  p.n_wtiles = wt;
  const int64_t total = static_cast<int64_t>(p.n_xtiles) * wt;
  if (total == 0) return CONVROT_OK;
  if (total > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
  p.total_tiles = static_cast<int>(total);
  p.n_lin = n_lin;
  p.raw_s32 = raw_s32 ? 1 : 0;

  static std::mutex mu;
  static uint64_t configured = 0;  // bit d: attribute set on device d
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 64 || !((configured >> dev) & 1u)) {
      cudaError_t e = cudaFuncSetAttribute(convrot_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
      if (e != cudaSuccess) return set_cuda_error(e);
      if (dev < 64) configured |= (1ull << dev);
    }
  }
  const int grid = static_cast<int>(std::min<int64_t>(total, device_sm_count()));
  convrot_gemm_kernel<<<grid, THREADS, SMEM_ALLOC, stream>>>(p);
  return check_launch();
}

int read_and_clear_device_error(cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return set_cuda_error(e);
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int));
  if (e != cudaSuccess) return set_cuda_error(e);
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
    if (e != cudaSuccess) return set_cuda_error(e);
  }
  return v;
}

}  // namespace convrot
