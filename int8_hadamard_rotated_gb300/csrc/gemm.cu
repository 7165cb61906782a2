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
// Kernel shape. Persistent, one CTA per SM, 10 warps:
//   warps 0-7  epilogue: drain TMEM chunks into registers, reconstruct, and
//              store through shared memory with tensor-map stores (each
//              thread owns one output feature o and 128 activation rows of a
//              tile).
//   warp 8     TMA producer: streams 64-deep K slices of the weight and
//              activation binary16 codes (128-byte swizzle) into a ring of
//              shared-memory stages.
//   warp 9     MMA issuer: one thread issues tcgen05.mma kind::f16 with
//              N = 256 activation rows and K = 16 into one of two 256-column
//              fp32 TMEM accumulators that alternate per K-chunk, so the
//              epilogue drains one while the other accumulates.
// Two variants, CG = CTAs per MMA:
//   CG = 2 (default): CTA pairs (clusters of two). A tile is 256 weight rows x
//     256 activation rows; each CTA loads 128 rows of each operand per stage
//     (32 KB, 6 stages) and holds the accumulator of its 128 weight rows. The
//     even CTA issues the pair's MMAs (M = 256) once both halves have landed on
//     its "full" barrier; commits arrive on both CTAs' barriers.
//   CG = 1: single CTAs, 128 weight rows x 256 activation rows per tile
//     (48 KB, 4 stages); used where clusters cannot be launched.
// Tiles of all linears sharing the input form one launch, walked so that the
// activation bands of a raster group stay in L2 while their weight tiles
// stream through; a fractional last wave can be split by K (split waves).
#include "gemm_common.cuh"

#include <cuda.h>
#include <algorithm>
#include <atomic>
#include <chrono>
#include <type_traits>
#include <mutex>

namespace convrot {

// Sticky device error word of the GEMM kernel (timeouts of bounded waits).
__device__ int g_device_error = 0;

namespace {

using namespace gemm;

constexpr int kActNone = 0;
constexpr int kActGelu = 1;
constexpr int kActSwiglu = 2;

// K blocks per exact chunk of a tile. For split SwiGLU the tile holds the
// features c.wt * 128 .. +127 of both weights, each one plan block: the
// shorter of the two plans' runs.
template <int CG, bool SWIGLU>
__device__ __forceinline__ int chunk_kb(const GemmParams& p, const TileCoord& c) {
  if (!SWIGLU) return tile_chunk_kb<CG>(p, c);
  int L = KB_PER_CHUNK;
  if (p.kchunk[0] && p.kchunk[1]) L = min(__ldg(p.kchunk[0] + c.wt), __ldg(p.kchunk[1] + c.wt));
  return max(1, min(L, p.num_kb));
}

// UNSCALE: the variant for linears with an input scale other than 1 (the IEEE
// division stays out of the common kernel's unrolled epilogue).
// YTMA: Y leaves through shared memory and tensor-map stores (Y_ROWS rows x
// 128 features per store) instead of per-thread global stores.
// ACT (CTA pairs with YTMA only): an activation applied to the reconstructed
// output before it is stored.
//   kActGelu: Y = gelu(y) elementwise.
//   kActSwiglu: split SwiGLU of two linears that share the input, gate
//     (linear 0) and up (linear 1) with the same N: a tile covers 128 output
//     features, and each CTA of the pair holds 64 of them in both weights
//     (rows 0-63 of its tile: gate, rows 64-127: up, loaded from the two
//     weight tensors as they are). The epilogue reconstructs both and writes
//     only h = silu(gate) * up, through a 64-feature staging tile.
template <int CG, int BN_, bool UNSCALE, bool YTMA, int ACT = kActNone>
__global__ void __launch_bounds__(THREADS, 1)
convrot_gemm_kernel(const __grid_constant__ GemmParams p) {
  static_assert(ACT == kActNone || (CG == 2 && YTMA && !UNSCALE), "activations: pair kernel, staged stores");
  constexpr bool SWIGLU = (ACT == kActSwiglu);
  using Gm = Geom<CG, BN_, YTMA>;
  constexpr int BN = Gm::BN;
  constexpr int COLS_PER_THREAD = Gm::COLS;
  constexpr int STAGES = Gm::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Gm::SMEM_BARS);
  uint64_t* full = bars;                   // [STAGES]
  uint64_t* empty = bars + STAGES;         // [STAGES]
  uint64_t* tfull = bars + 2 * STAGES;     // [2]
  uint64_t* tempty = bars + 2 * STAGES + 2;
  uint64_t* drain = bars + 2 * STAGES + 4;
  uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(smem + Gm::SMEM_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Gm::SMEM_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int* err = &g_device_error;
  constexpr int UNIT_CTAS = CG;  // CTAs per scheduling unit (a pair or a CTA)
  // CTA rank in its pair (0 issues the pair's MMAs) and the scheduling unit
  const uint32_t crank = (CG == 2) ? cluster_ctarank() : 0u;
  const uint32_t rank = crank;
  const uint32_t lead_rank = 0u;  // the pair leader's rank in the cluster
  const bool leader = (rank == 0);
  const int unit = (CG == 2) ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int n_units = (CG == 2) ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);
  // the pair's CTAs: a pair's MMA commits arrive on both
  const uint16_t pair_mask = 0x3u;

  if (threadIdx.x == PRODUCER_WARP * 32) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], NUM_EPI_WARPS * CG);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&p.tmap_x);
    for (int j = 0; j < p.n_lin; ++j) tma_prefetch_desc(&p.tmap_w[j]);
  }
  if (warp == MMA_WARP) {
    if (CG == 2) {
      tmem_alloc_pair(tmem_base_smem, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_base_smem, TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (CG == 2) cluster_sync(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_smem;
  // Launched as a programmatic dependent of the kernel before it (the pack):
  // everything above overlapped that kernel; nothing below may read or write
  // global memory before it has completed.
  pdl_wait_prerequisites();

  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      const uint64_t pol_x = l2_policy_evict_normal();
      const uint64_t pol_w = l2_policy_evict_normal();
      // the pair's "full" barriers live in the leader CTA
      const uint32_t full_leader = (CG == 2) ? mapa_shared(smem_u32(full), lead_rank) : smem_u32(full);
      uint32_t stage = 0, phase = 0;
      uint32_t n_issued = 0;  // stage loads issued so far (stage = n % STAGES)
      bool ok = true;
      WorkItem it;
      for (int j = 0; ok && work_item(p, unit, n_units, j, it); ++j) {
        const TileCoord c = decode_tile(p, it.t);
        const int w_row = c.wt * Gm::TILE_M + static_cast<int>(rank) * CTA_M;
        const int x_row = c.xt * BN + static_cast<int>(rank) * Gm::X_ROWS;
        for (int kb = it.kb0; kb < it.kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err, p.wait_ns)) { ok = false; break; }
          uint8_t* sw = smem + stage * Gm::STAGE_BYTES;
          uint8_t* sx = sw + Gm::W_BYTES;
          if (CG == 2) {
            if (leader) mbar_arrive_expect_tx(&full[stage], CG * Gm::STAGE_BYTES);
            const uint32_t fb = full_leader + stage * 8u;
            if (SWIGLU) {
              // this CTA's 64 features of the gate weight, then of the up weight
              const int f = c.wt * 128 + static_cast<int>(rank) * 64;
              tma_load_2d_pair(sw, &p.tmap_w[0], fb, kb * BK, f, pol_w);
              tma_load_2d_pair(sw + 64 * BK * 2, &p.tmap_w[1], fb, kb * BK, f, pol_w);
            } else {
              tma_load_2d_pair(sw, &p.tmap_w[c.lin], fb, kb * BK, w_row, pol_w);
            }
            tma_load_2d_pair(sx, &p.tmap_x, fb, kb * BK, x_row, pol_x);
          } else {
            mbar_arrive_expect_tx(&full[stage], Gm::STAGE_BYTES);
            tma_load_2d(sw, &p.tmap_w[c.lin], &full[stage], kb * BK, w_row, pol_w);
            tma_load_2d(sx, &p.tmap_x, &full[stage], kb * BK, x_row, pol_x);
          }
          ++n_issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // No copy may land after the CTAs exit: the leader waits (bounded) for
      // the last phase of every stage that was ever filled (its barriers count
      // both CTAs' bytes); the pair then meets at the final cluster barrier.
      if (leader)
        for (uint32_t s = 0; s < STAGES; ++s)
          if (n_issued > s) {
            const uint32_t uses = (n_issued - 1 - s) / STAGES + 1;  // times stage s was filled
            mbar_wait(&full[s], (uses - 1) & 1u, nullptr, err, p.wait_ns);
          }
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    if (lane == 0 && leader) {
      uint32_t stage = 0, phase = 0, chunk_iter = 0;
      bool ok = true;
      // the next item's chunk length is read one item ahead
      WorkItem it, nx;
      int j = 0;
      bool have = work_item(p, unit, n_units, j, it);
      int L = have ? chunk_kb<CG, SWIGLU>(p, decode_tile(p, it.t)) : 1;
      while (ok && have) {
        const bool have_nx = work_item(p, unit, n_units, ++j, nx);
        const int L_nx = have_nx ? chunk_kb<CG, SWIGLU>(p, decode_tile(p, nx.t)) : 1;
        for (int c0 = it.kb0; ok && c0 < it.kb1;) {
          const int c1 = chunk_end(c0, L, it.kb1);
          const uint32_t buf = chunk_iter & 1u;
          const uint32_t use = chunk_iter >> 1;
          if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort_flag, err, p.wait_ns)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * BN;
          const int kb0 = c0;
          const int kb1 = c1;
          c0 = c1;
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(&full[stage], phase, abort_flag, err, p.wait_ns)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sw = smem_u32(smem + stage * Gm::STAGE_BYTES);
            const uint64_t a_desc = smem_desc_sw128(sw);
            const uint64_t b_desc = smem_desc_sw128(sw + Gm::W_BYTES);
#pragma unroll
            for (int k = 0; k < BK / UMMA_K; ++k) {
              // advance the start address by k * 32 bytes inside the swizzle row
              const uint64_t koff = static_cast<uint64_t>((k * UMMA_K * 2) >> 4);
              const uint32_t acc = (kb > kb0 || k > 0) ? 1u : 0u;
              if (CG == 2) mma_f16_ss_pair(d_tmem, a_desc + koff, b_desc + koff, Gm::IDESC, acc);
              else mma_f16_ss(d_tmem, a_desc + koff, b_desc + koff, Gm::IDESC, acc);
            }
            if (CG == 2) mma_commit_pair(&empty[stage], pair_mask); else mma_commit(&empty[stage]);
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          if (CG == 2) mma_commit_pair(&tfull[buf], pair_mask); else mma_commit(&tfull[buf]);
          ++chunk_iter;
        }
        it = nx;
        L = L_nx;
        have = have_nx;
      }
      // all issued MMAs complete before TMEM is released
      if (CG == 2) mma_commit_pair(drain, static_cast<uint16_t>(1u << lead_rank)); else mma_commit(drain);
      mbar_wait(drain, 0, nullptr, err, p.wait_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------ epilogue ------------------------------
    const uint64_t pol_y = l2_policy_evict_first();
    const int quarter = warp & 3;             // TMEM lanes 32*quarter .. +31
    const int half = warp >> 2;               // activation columns half*128 .. +127
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    // the pair's "accumulator free" barriers live in the leader CTA
    const uint32_t tempty_leader = (CG == 2) ? mapa_shared(smem_u32(tempty), lead_rank) : smem_u32(tempty);
    uint32_t chunk_iter = 0;
    bool ok = true;
    WorkItem it;
    for (int j = 0; ok && work_item(p, unit, n_units, j, it); ++j) {
      const TileCoord c = decode_tile(p, it.t);
      const int L = chunk_kb<CG, SWIGLU>(p, c);
      // One exact chunk (the whole K of a tile that is not split) is kept as
      // the fp32 value TMEM holds: an integer below 2^24, so it is float(A)
      // itself. Several chunks, a split tile and the raw int32 output add the
      // chunks in int32 first.
      const int n_chunks = (it.kb1 - 1) / L - it.kb0 / L + 1;
      const bool int_path = p.raw_s32 || n_chunks > 1 || it.kind != kWhole;
      int acc[COLS_PER_THREAD];
#pragma unroll
      for (int i = 0; i < COLS_PER_THREAD; ++i) acc[i] = 0;
      for (int c0 = it.kb0; c0 < it.kb1; c0 = chunk_end(c0, L, it.kb1)) {
        const uint32_t buf = chunk_iter & 1u;
        const uint32_t use = chunk_iter >> 1;
        if (!mbar_wait(&tfull[buf], use & 1u, abort_flag, err, p.wait_ns)) { ok = false; break; }
        tc_fence_after();
        if (int_path) {
#pragma unroll
          for (int q = 0; q < COLS_PER_THREAD / 32; ++q) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tmem_base + lane_base + buf * BN + half * COLS_PER_THREAD + q * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[q * 32 + i] += __float2int_rz(__uint_as_float(r[i]));
          }
        } else {
#pragma unroll
          for (int q = 0; q < COLS_PER_THREAD / 32; ++q) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tmem_base + lane_base + buf * BN + half * COLS_PER_THREAD + q * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[q * 32 + i] = static_cast<int>(r[i]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (CG == 2) mbar_arrive_cluster(tempty_leader + buf * 8u);
          else mbar_arrive(&tempty[buf]);
        }
        ++chunk_iter;
      }
      // the eight epilogue warps leave together (the Y stores and the hand-over
      // of split tiles use barriers of their own)
      ok = named_bar_and(EPI_BAR, NUM_EPI_WARPS * 32, ok);
      if (!ok) break;
      const int N = p.N[c.lin];
      // the output feature of this thread's TMEM lane (split SwiGLU: lanes
      // 0-63 hold the gate and 64-127 the up weight of the CTA's 64 features)
      const int o = SWIGLU ? c.wt * 128 + static_cast<int>(rank) * 64 + ((32 * quarter + lane) & 63)
                           : c.wt * Gm::TILE_M + static_cast<int>(rank) * CTA_M + 32 * quarter + lane;
      const int wsel = (SWIGLU && 32 * quarter + lane >= 64) ? 1 : c.lin;  // the linear whose scale and bias apply
      const bool o_ok = o < N;
      const int r0 = c.xt * BN + half * COLS_PER_THREAD;
      // partial sums of a split tile travel through the tile's own output, as int32
      int32_t* part = static_cast<int32_t*>(p.out[c.lin]);
      if (it.kind == kHead) {
        if (o_ok) {
#pragma unroll
          for (int i = 0; i < COLS_PER_THREAD; ++i) {
            const int r = r0 + i;
            if (r < p.M) part[static_cast<int64_t>(r) * N + o] = acc[i];
          }
        }
        __threadfence();
        named_bar_sync(EPI_BAR, NUM_EPI_WARPS * 32);
        if (threadIdx.x == 0) st_release_gpu(p.sk_flags + UNIT_CTAS * unit + crank, p.epoch);
        continue;
      }
      if (it.kind == kTail) {
        bool got = true;
        if (threadIdx.x == 0) {
          unsigned long long* f = p.sk_flags + UNIT_CTAS * (unit - 1) + crank;
          got = wait_flag(f, p.epoch ^ p.handover_xor, abort_flag, err, p.wait_ns);
          if (got) st_relaxed_gpu(f, 0ull);  // consumed: zero again for the next launch
        }
        ok = named_bar_and(EPI_BAR, NUM_EPI_WARPS * 32, got);
        if (!ok) break;
        if (o_ok) {
          // 16 loads in flight at a time (L2 only: the partial sums were
          // written by another SM)
#pragma unroll
          for (int q = 0; q < COLS_PER_THREAD / 16; ++q) {
            int32_t v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int r = r0 + 16 * q + i;
              v[i] = (r < p.M) ? __ldcg(part + static_cast<int64_t>(r) * N + o) : 0;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[16 * q + i] += v[i];
          }
        }
      }
      if (p.raw_s32) {
        if (o_ok) {
          int32_t* A = static_cast<int32_t*>(p.out[c.lin]);
#pragma unroll
          for (int i = 0; i < COLS_PER_THREAD; ++i) {
            const int r = r0 + i;
            if (r < p.M) st_global_hint(A + static_cast<int64_t>(r) * N + o, acc[i], pol_y);
          }
        }
      } else {
        // from here acc holds float(A) as fp32 bits (the int32 sum rounded to nearest)
        if (int_path) {
#pragma unroll
          for (int i = 0; i < COLS_PER_THREAD; ++i) acc[i] = __float_as_int(__int2float_rn(acc[i]));
        }
        // the warp's 128 row scales: four per lane, broadcast by shuffles
        // (YTMA: the warpgroup's row scales staged in shared memory instead)
        float sxv[COLS_PER_THREAD / 32];
        if (!YTMA) {
#pragma unroll
          for (int k = 0; k < COLS_PER_THREAD / 32; ++k) {
            const int r = r0 + 32 * k + lane;
            sxv[k] = (r < p.M) ? __ldg(p.s_x + r) : 0.0f;
          }
        }
        float* Y = static_cast<float*>(p.out[c.lin]);
        const float* sw_ptr = p.s_w[wsel];
        const float* b_ptr = p.bias[wsel];
        const float sw = (o_ok && sw_ptr) ? __ldg(sw_ptr + o) : 1.0f;
        const float bb = (o_ok && b_ptr) ? __ldg(b_ptr + o) : 0.0f;
        const float in_scale = UNSCALE ? p.in_scale[c.lin] : 1.0f;
        if (YTMA) {
          // Y_ROWS rows at a time through this warpgroup's two staging
          // buffers in turn and one tensor-map store each (rows past M and
          // features past N are not written by the store)
          uint8_t* sy_base = smem + Gm::SMEM_YOUT + half * Y_HALF_BYTES;
          const bool store_leader = (quarter == 0 && lane == 0);
          const int col = 32 * quarter + lane;
          const int o_base = c.wt * Gm::TILE_M + static_cast<int>(rank) * CTA_M;
          const unsigned long long sw2 = pair_f32(sw, sw), bb2 = pair_f32(bb, bb);
          // the warpgroup's row scales, read back four at a time (a broadcast:
          // every lane reads the same address); the first barrier below orders
          // the writes before the reads, and the previous tile's reads ended
          // before the epilogue-wide barrier of this tile
          float* ssx = reinterpret_cast<float*>(smem + Gm::SMEM_SX) + half * 128;
          if (col < COLS_PER_THREAD) ssx[col] = (r0 + col < p.M) ? __ldg(p.s_x + r0 + col) : 0.0f;
          // unscaling: the tile's extreme row scales decide, per thread,
          // whether the correction step may replace the division
          Unscale us{};
          bool us_fast = false;
          if (UNSCALE) {
            named_bar_sync(1 + half, 4 * 32);
            float v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) v[k] = (lane + 32 * k < COLS_PER_THREAD) ? ssx[lane + 32 * k] : 0.0f;
            float lo, hi;
            warp_scale_range(v, lo, hi);
            us = make_unscale(in_scale);
            us_fast = unscale_fast_ok(in_scale, lo, hi, sw);
          }
          const unsigned long long m1 = pair_f32(-1.0f, -1.0f);
          // The row blocks, once with the correction step (FAST) and once with
          // the IEEE division, so that the loop that runs is contiguous code
          // (unrolled so that the accumulators stay in registers).
          auto row_blocks = [&](auto fast_tag) {
            constexpr bool FAST = decltype(fast_tag)::value;
#pragma unroll
            for (int sub = 0; sub < COLS_PER_THREAD / Y_ROWS; ++sub) {
              // every block commits one bulk group (empty when nothing is
              // stored) and the count of blocks per tile is even, so the group
              // two back is the last store from this buffer: wait until it read it
              // (split SwiGLU: y is staged in buffer 0, reused every block, and
              // h in one half of buffer 1 per block, the half two blocks back
              // being the last one stored)
              float* sy = reinterpret_cast<float*>(sy_base + (SWIGLU ? 0 : (sub & 1) * Y_BUF_BYTES));
              if (store_leader) bulk_wait_read<1>();
              named_bar_sync(1 + half, 4 * 32);
#pragma unroll
              for (int i = 0; i < Y_ROWS; i += 4) {
                const int idx = sub * Y_ROWS + i;
                const float4 s4 = *reinterpret_cast<const float4*>(ssx + idx);
                // float(A) * s_x * s_w (/ input scale) + b, one rounding per
                // operation, in that order, two rows at once
                unsigned long long ya = mul_f32x2(pair_f32(__int_as_float(acc[idx]), __int_as_float(acc[idx + 1])),
                                                  pair_f32(s4.x, s4.y));
                unsigned long long yb = mul_f32x2(pair_f32(__int_as_float(acc[idx + 2]), __int_as_float(acc[idx + 3])),
                                                  pair_f32(s4.z, s4.w));
                if (sw_ptr) {
                  ya = mul_f32x2(ya, sw2);
                  yb = mul_f32x2(yb, sw2);
                }
                if (UNSCALE && FAST) {
                  // unscale before the bias: -RN(y / a) by the correction step,
                  // then RN(b - (-q)) or -(-q)
                  ya = neg_unscale_f32x2(ya, us);
                  yb = neg_unscale_f32x2(yb, us);
                  if (b_ptr) {
                    ya = f32x2_fma(ya, m1, bb2);
                    yb = f32x2_fma(yb, m1, bb2);
                  } else {
                    ya = mul_f32x2(ya, m1);
                    yb = mul_f32x2(yb, m1);
                  }
                } else {
                  if (UNSCALE && !FAST) {
                    // unscale before the bias (IEEE division, element by element)
                    ya = unscale_div_f32x2(ya, in_scale);
                    yb = unscale_div_f32x2(yb, in_scale);
                  }
                  if (b_ptr) {
                    ya = add_f32x2(ya, bb2);
                    yb = add_f32x2(yb, bb2);
                  }
                }
                float y0, y1, y2, y3;
                unpair_f32(ya, y0, y1);
                unpair_f32(yb, y2, y3);
                if (ACT == kActGelu) {
                  gelu_as2(y0, y1);
                  gelu_as2(y2, y3);
                }
                sy[i * CTA_M + col] = y0;
                sy[(i + 1) * CTA_M + col] = y1;
                sy[(i + 2) * CTA_M + col] = y2;
                sy[(i + 3) * CTA_M + col] = y3;
              }
              // Split SwiGLU: the product is evaluated by the warps of TMEM
              // quarters 2 and 3 only (quarter 0 shares its scheduler with the
              // TMA producer and quarter 1 with the MMA issuer, which pace the
              // kernel), eight independent rows per thread.
              const int awork = col - 64;  // 0 .. 63 in quarters 2 and 3
              if (SWIGLU) {
                // h = silu(gate) * up for the CTA's 64 features: gate in staged
                // columns 0-63, up in 64-127
                named_bar_sync(1 + half, 4 * 32);
                float* sh = reinterpret_cast<float*>(sy_base + Y_BUF_BYTES) + (sub & 1) * (Y_ROWS * 64);
                if (awork >= 0) {
#pragma unroll
                  for (int i = 0; i < Y_ROWS; ++i)
                    sh[i * 64 + awork] = silu_mul_fast(sy[i * CTA_M + awork], sy[i * CTA_M + 64 + awork]);
                }
                fence_proxy_async_smem();
                named_bar_sync(1 + half, 4 * 32);
                if (store_leader) {
                  const int f0 = c.wt * 128 + static_cast<int>(rank) * 64;
                  if (f0 < N && r0 + sub * Y_ROWS < p.M) tma_store_2d(&p.tmap_y[0], sh, f0, r0 + sub * Y_ROWS);
                  bulk_commit();
                }
              } else {
                fence_proxy_async_smem();
                named_bar_sync(1 + half, 4 * 32);
                if (store_leader) {
                  if (o_base < N && r0 + sub * Y_ROWS < p.M) tma_store_2d(&p.tmap_y[c.lin], sy, o_base, r0 + sub * Y_ROWS);
                  bulk_commit();
                }
              }
            }
          };
          if (!UNSCALE || us_fast) row_blocks(std::true_type{});
          else row_blocks(std::false_type{});
        } else {
          Unscale us{};
          bool us_fast = false;
          if (UNSCALE) {
            float lo, hi;
            warp_scale_range(sxv, lo, hi);
            us = make_unscale(in_scale);
            us_fast = unscale_fast_ok(in_scale, lo, hi, sw);
          }
#pragma unroll
          for (int i = 0; i < COLS_PER_THREAD; ++i) {
            const float sx = __shfl_sync(0xffffffffu, sxv[i >> 5], i & 31);
            const int r = r0 + i;
            if (o_ok && r < p.M) {
              // float(A) * s_x * s_w + b, one rounding per operation, in that order
              float y = __fmul_rn(__int_as_float(acc[i]), sx);
              if (sw_ptr) y = __fmul_rn(y, sw);
              // unscale before the bias
              if (UNSCALE) y = us_fast ? -neg_unscale_f32(y, us) : __fdiv_rn(y, in_scale);
              if (b_ptr) y = __fadd_rn(y, bb);
              st_global_hint(Y + static_cast<int64_t>(r) * N + o, y, pol_y);
            }
          }
        }
      }
    }
    // the last tensor-map stores complete before the CTA releases its shared memory
    if (YTMA && (warp & 3) == 0 && lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  if (CG == 2) cluster_sync(); else __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    if (CG == 2) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

template <int CG, int BN>
int fill_params(GemmParams& p, const __half* x16, const float* s_x, int64_t M, int64_t K,
                const GemmLinear* lins, int n_lin, bool raw_s32) {
  using Gm = Geom<CG, BN>;
  memset(&p, 0, sizeof(p));
  int st = make_tmap(&p.tmap_x, x16, M, K, Gm::X_ROWS);
  if (st) return st;
  int wt = 0;
  for (int j = 0; j < n_lin; ++j) {
    st = make_tmap(&p.tmap_w[j], lins[j].w16, lins[j].N, K, CTA_M);
    if (st) return st;
    p.s_w[j] = lins[j].s_w;
    p.bias[j] = lins[j].bias;
    p.kchunk[j] = lins[j].kchunk;
    p.in_scale[j] = lins[j].in_scale;
    p.out[j] = lins[j].out;
    p.N[j] = static_cast<int>(lins[j].N);
    p.wtile_start[j] = wt;
    wt += static_cast<int>((lins[j].N + Gm::TILE_M - 1) / Gm::TILE_M);
  }
  p.wtile_start[n_lin] = wt;
  p.s_x = s_x;
  p.M = static_cast<int>(M);
  p.K = static_cast<int>(K);
  p.num_kb = static_cast<int>((K + BK - 1) / BK);
  p.n_xtiles = static_cast<int>((M + BN - 1) / BN);
  p.n_wtiles = wt;
  const int64_t band_bytes = static_cast<int64_t>(BN) * K * 2;
  p.raster_bands = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(p.n_xtiles, RASTER_L2_BYTES / band_bytes)));
  const int64_t total = static_cast<int64_t>(p.n_xtiles) * wt;
  if (total > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
  p.total_tiles = static_cast<int>(total);
  p.n_lin = n_lin;
  p.raw_s32 = raw_s32 ? 1 : 0;
  p.sk_tiles = 0;
  p.wait_ns = kWaitLimitNs;
  p.handover_xor = 0;
  return CONVROT_OK;
}

template <int CG, int BN, bool UNSCALE, bool YTMA, int ACT = kActNone>
int configure_kernel() {
  static std::mutex mu;
  static uint64_t configured = 0;  // bit d: attribute set on device d
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_cuda_error(e);
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 64 || !((configured >> dev) & 1u)) {
    e = cudaFuncSetAttribute(convrot_gemm_kernel<CG, BN, UNSCALE, YTMA, ACT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, Geom<CG, BN, YTMA>::SMEM_ALLOC);
    if (e != cudaSuccess) return set_cuda_error(e);
    if (dev < 64) configured |= (1ull << dev);
  }
  return CONVROT_OK;
}

// Co-resident CTA pairs of the BN variant on the current device (0 if they
// cannot launch), cached per device. The kernel must be configured first.
template <int BN>
int max_pairs() {
  static std::mutex mu;
  static int cached[64];
  static bool known[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!known[dev]) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pair_config(device_sm_count() / 2, Geom<2, BN, true>::SMEM_ALLOC, nullptr, attr, false);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, convrot_gemm_kernel<2, BN, false, true>, &cfg) != cudaSuccess) {
      cudaGetLastError();  // clear the sticky launch-query error
      n = 0;
    }
    cached[dev] = n;
    known[dev] = true;
  }
  return cached[dev];
}

// `pairs`: co-resident CTA pairs of the variant.
template <int BN, bool UNSCALE, bool YTMA>
int launch_pairs(const __half* x16, const float* s_x, int64_t M, int64_t K, const GemmLinear* lins, int n_lin,
                 bool raw_s32, int pairs, cudaStream_t stream, const GemmSync& sync) {
  GemmParams p;
  if (int st = fill_params<2, BN>(p, x16, s_x, M, K, lins, n_lin, raw_s32)) return st;
  if (p.total_tiles == 0) return CONVROT_OK;
  if (YTMA)
    for (int j = 0; j < n_lin; ++j)
      if (int st = make_tmap_y(&p.tmap_y[j], lins[j].out, M, lins[j].N, CTA_M)) return st;
  const int units = std::min(p.total_tiles, pairs);
  if (BN == 256) plan_split(p, units, 2, sync);
  if (sync.test_wait_ns) p.wait_ns = sync.test_wait_ns;
  if (sync.test_unpublished_handover) p.handover_xor = 1;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = pair_config(units, Geom<2, BN, YTMA>::SMEM_ALLOC, stream, attr, true);
  if (int st = configure_kernel<2, BN, UNSCALE, YTMA>()) return st;
  cudaError_t e = cudaLaunchKernelEx(&cfg, convrot_gemm_kernel<2, BN, UNSCALE, YTMA>, p);
  if (e != cudaSuccess) return set_cuda_error(e);
  return check_launch();
}

// ---------------------------------------------------------------------------
// exact-chunk plan of a weight (offline)
// ---------------------------------------------------------------------------

constexpr int kPlanMaxCands = 16;
constexpr long long kExactLimit = (1ll << 24) - 1;  // every integer up to this is exact in fp32

// One thread per weight row, one CTA per block of CONVROT_CHUNK_ROWS rows.
// Candidates: runs of 16 * 2^j K blocks (shorter than K), then all of K. For
// each candidate, the largest 127 * sum |Q_w| over any run of any row of the
// block decides whether the candidate is exact.
__global__ void __launch_bounds__(CONVROT_CHUNK_ROWS)
chunk_plan_kernel(const int8_t* __restrict__ Q_w, int N, int K, int32_t* __restrict__ kchunk) {
  const int num_kb = (K + BK - 1) / BK;
  int cand[kPlanMaxCands];
  int nc = 0;
  for (int L = KB_PER_CHUNK; L < num_kb && nc < kPlanMaxCands - 1; L *= 2) cand[nc++] = L;
  cand[nc++] = num_kb;
  int run[kPlanMaxCands], mx[kPlanMaxCands];
  for (int c = 0; c < nc; ++c) run[c] = mx[c] = 0;
  const int o = blockIdx.x * CONVROT_CHUNK_ROWS + threadIdx.x;
  if (o < N) {
    const int8_t* row = Q_w + static_cast<int64_t>(o) * K;
    for (int kb = 0; kb < num_kb; ++kb) {
      int sum = 0;
      const int e1 = min(K, (kb + 1) * BK);
      for (int e = kb * BK; e < e1; e += 16) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + e);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int b = 0; b < 4; ++b) sum += abs(static_cast<int>(static_cast<int8_t>((w[i] >> (8 * b)) & 0xffu)));
      }
      for (int c = 0; c < nc; ++c) {
        if (kb % cand[c] == 0) run[c] = 0;
        run[c] += sum;
        mx[c] = max(mx[c], run[c]);
      }
    }
  }
  __shared__ int s_max[kPlanMaxCands];
  if (threadIdx.x < kPlanMaxCands) s_max[threadIdx.x] = 0;
  __syncthreads();
  for (int c = 0; c < nc; ++c) atomicMax(&s_max[c], mx[c]);
  __syncthreads();
  if (threadIdx.x == 0) {
    int best = min(KB_PER_CHUNK, num_kb);  // 1024 products: always exact
    for (int c = 0; c < nc; ++c)
      if (static_cast<long long>(s_max[c]) * 127 <= kExactLimit) best = max(best, cand[c]);
    kchunk[blockIdx.x] = best;
  }
}

}  // namespace

namespace gemm {

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

// fp32 Y [rows, cols] row-major (cols % 4 == 0), box 128 features x Y_ROWS rows, no swizzle.
int make_tmap_y(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_cols) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return set_cuda_error(cudaErrorNotSupported);
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(Y_ROWS)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_cuda_error(cudaErrorInvalidValue);
  return CONVROT_OK;
}

// Nonzero value distinct per launch for the hand-over flags: a process-wide
// counter that starts at the wall clock in nanoseconds, so that flag words
// left in reused scratch by an earlier launch or process never match.
unsigned long long next_epoch() {
  static std::atomic<unsigned long long> counter{
      static_cast<unsigned long long>(std::chrono::duration_cast<std::chrono::nanoseconds>(
                                          std::chrono::system_clock::now().time_since_epoch())
                                          .count()) |
      1ull};
  return counter.fetch_add(1);
}

// Whole tiles only, or split tiles first, for `units` co-resident units. The
// split takes the fractional wave and one whole wave (so that every unit's
// range covers at least one tile) and is used only where it pays on this
// GPU: when a last wave of whole tiles would leave at least 40 % of the units
// idle and at least one whole wave remains after the split. (A last wave
// that is busier runs nearly as fast as the split: with fewer tiles in
// flight each runs faster. Splitting every tile adds the partial-sum
// hand-over to the end of the kernel.)
bool split_pays(int T, int units) {
  if (units < 2 || T < 2 * units) return false;
  const int rem = T % units;
  return rem != 0 && 10 * (units - rem) >= 4 * units;
}

void plan_split(GemmParams& p, int units, int unit_ctas, const GemmSync& sync) {
  p.sk_tiles = 0;
  const int T = p.total_tiles;
  if (!sync.words || sync.bytes < static_cast<size_t>(unit_ctas * units) * sizeof(unsigned long long)) return;
  if (!split_pays(T, units)) return;
  const int rem = T % units;
  p.sk_tiles = units + rem;
  p.sk_flags = sync.words;
  p.epoch = next_epoch();
}

// Raise the kernel's shared-memory limit once per device.
// Launch configuration of the CTA-pair kernel: n_units clusters of two CTAs
// and, when `pdl`, programmatic serialization after the previous kernel in
// the stream (the kernel waits for it with griddepcontrol.wait after its own
// setup).
cudaLaunchConfig_t pair_config(int n_units, size_t smem, cudaStream_t stream, cudaLaunchAttribute* attr,
                               bool pdl) {
  constexpr int cluster = 2;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster * n_units, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cfg;
}

}  // namespace gemm

int launch_chunk_plan(const int8_t* Q_w, int64_t N, int64_t K, int32_t* kchunk, cudaStream_t stream) {
  if (N == 0) return CONVROT_OK;
  const int64_t blocks = (N + CONVROT_CHUNK_ROWS - 1) / CONVROT_CHUNK_ROWS;
  chunk_plan_kernel<<<static_cast<unsigned>(blocks), CONVROT_CHUNK_ROWS, 0, stream>>>(
      Q_w, static_cast<int>(N), static_cast<int>(K), kchunk);
  return check_launch();
}

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

// Activation rows per tile: the tile height among 256, 192 and 128 with the
// least modelled time, waves x (BN + 96), where waves counts a partial last
// wave as a whole one unless the split will balance it (256-row tiles; then
// the fraction counts), and 96 stands for the cost of a tile that does not
// shrink with its height (the weight rows it streams); ties go to the taller
// tile.
int pick_tile_rows(int64_t M, const GemmLinear* lins, int n_lin, int pairs, bool can_split) {
  int64_t wtiles = 0;
  for (int j = 0; j < n_lin; ++j) wtiles += (lins[j].N + 2 * CTA_M - 1) / (2 * CTA_M);
  int best = 256;
  double best_cost = -1.0;
  for (int bn : {256, 192, 128}) {
    const int64_t tiles = ((M + bn - 1) / bn) * wtiles;
    // only 256-row tiles are split (shorter tiles lose more than the split gains)
    const bool split = can_split && bn == 256 && tiles <= 0x7fffffff && split_pays(static_cast<int>(tiles), pairs);
    const double waves = split ? static_cast<double>(tiles) / pairs : static_cast<double>((tiles + pairs - 1) / pairs);
    const double cost = waves * (bn + 96);
    if (best_cost < 0.0 || cost < best_cost) { best = bn; best_cost = cost; }
  }
  return best;
}

namespace {

// The activation variants: 256-row pair tiles with staged stores. GELU takes
// the linears as usual (and may split its last wave); split SwiGLU takes
// lins[0] (gate) and lins[1] (up), same N, whole tiles only (a split tile's
// partial sums of both weights would need twice the output's room), and
// writes h to lins[0].out.
template <int ACT>
int launch_act(const __half* x16, const float* s_x, int64_t M, int64_t K, const GemmLinear* lins, int n_lin,
               int pairs, cudaStream_t stream, const GemmSync& sync) {
  constexpr int BN = 256;
  GemmParams p;
  if (ACT == kActSwiglu) {
    if (n_lin != 2 || lins[0].N != lins[1].N) return CONVROT_ERR_ARG;
    if (int st = fill_params<2, BN>(p, x16, s_x, M, K, lins, 1, false)) return st;
    // both weights in boxes of 64 rows; one tile per 128 features
    if (int st = make_tmap(&p.tmap_w[0], lins[0].w16, lins[0].N, K, 64)) return st;
    if (int st = make_tmap(&p.tmap_w[1], lins[1].w16, lins[1].N, K, 64)) return st;
    for (int j = 0; j < 2; ++j) {
      p.s_w[j] = lins[j].s_w;
      p.bias[j] = lins[j].bias;
      p.kchunk[j] = lins[j].kchunk;
    }
    const int wt = static_cast<int>((lins[0].N + 127) / 128);
    p.wtile_start[0] = 0;
    p.wtile_start[1] = wt;
    p.n_wtiles = wt;
    const int64_t total = static_cast<int64_t>(p.n_xtiles) * wt;
    if (total > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
    p.total_tiles = static_cast<int>(total);
    if (int st = make_tmap_y(&p.tmap_y[0], lins[0].out, M, lins[0].N, 64)) return st;
  } else {
    if (int st = fill_params<2, BN>(p, x16, s_x, M, K, lins, n_lin, false)) return st;
    for (int j = 0; j < n_lin; ++j)
      if (int st = make_tmap_y(&p.tmap_y[j], lins[j].out, M, lins[j].N, CTA_M)) return st;
  }
  if (p.total_tiles == 0) return CONVROT_OK;
  const int units = std::min(p.total_tiles, pairs);
  if (ACT != kActSwiglu) plan_split(p, units, 2, sync);
  if (int st = configure_kernel<2, BN, false, true, ACT>()) return st;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = pair_config(units, Geom<2, BN, true>::SMEM_ALLOC, stream, attr, true);
  cudaError_t e = cudaLaunchKernelEx(&cfg, convrot_gemm_kernel<2, BN, false, true, ACT>, p);
  if (e != cudaSuccess) return set_cuda_error(e);
  return check_launch();
}

}  // namespace

int launch_gemm_act(const __half* x16, const float* s_x, int64_t M, int64_t K, const GemmLinear* lins, int n_lin,
                    int act, cudaStream_t stream, GemmSync sync) {
  if (M == 0) return CONVROT_OK;
  if (act == CONVROT_ACT_NONE) return launch_linears(x16, s_x, M, K, lins, n_lin, false, stream, sync);
  bool w4 = false;
  for (int j = 0; j < n_lin; ++j) {
    if (lins[j].N % 4 != 0) return CONVROT_ERR_ALIGN;
    if (lins[j].in_scale != 1.0f) return CONVROT_ERR_UNSUPPORTED;
    w4 |= !lins[j].w16;
  }
  if (w4) {
    // packed 4-bit weights: GELU in the S8 x S4 GEMM's epilogue (every linear W4)
    if (act != CONVROT_ACT_GELU) return CONVROT_ERR_UNSUPPORTED;
    for (int j = 0; j < n_lin; ++j)
      if (lins[j].w16) return CONVROT_ERR_UNSUPPORTED;
    return launch_gemm_w4(x16, s_x, M, K, lins, n_lin, false, stream, sync, true);
  }
  if (int st = configure_kernel<2, 256, false, true>()) return st;
  const int pairs = max_pairs<256>();
  if (pairs <= 0) return CONVROT_ERR_UNSUPPORTED;
  if (act == CONVROT_ACT_GELU) return launch_act<kActGelu>(x16, s_x, M, K, lins, n_lin, pairs, stream, sync);
  if (act == CONVROT_ACT_SWIGLU) return launch_act<kActSwiglu>(x16, s_x, M, K, lins, n_lin, pairs, stream, sync);
  return CONVROT_ERR_ARG;
}

int launch_gemm(const __half* x16, const float* s_x, int64_t M, int64_t K,
                const GemmLinear* lins, int n_lin, bool raw_s32, cudaStream_t stream, GemmSync sync) {
  if (M == 0) return CONVROT_OK;
  bool unscale = false, ytma = !raw_s32;
  for (int j = 0; j < n_lin; ++j) {
    unscale |= (lins[j].in_scale != 1.0f);
    ytma &= (lins[j].N % 4 == 0);  // tensor-map rows must be multiples of 16 bytes
  }
  if (int st = configure_kernel<2, 256, false, true>()) return st;
  if (int st = configure_kernel<2, 192, false, true>()) return st;
  if (int st = configure_kernel<2, 128, false, true>()) return st;
  const int pairs = std::min(max_pairs<256>(), std::min(max_pairs<192>(), max_pairs<128>()));
  if (pairs > 0) {
    const bool can_split = sync.words && sync.bytes >= static_cast<size_t>(2 * pairs) * sizeof(unsigned long long);
    const int bn = pick_tile_rows(M, lins, n_lin, pairs, can_split);
    if (ytma && unscale) {
      if (bn == 128) return launch_pairs<128, true, true>(x16, s_x, M, K, lins, n_lin, raw_s32, pairs, stream, sync);
      if (bn == 192) return launch_pairs<192, true, true>(x16, s_x, M, K, lins, n_lin, raw_s32, pairs, stream, sync);
      return launch_pairs<256, true, true>(x16, s_x, M, K, lins, n_lin, raw_s32, pairs, stream, sync);
    }
    if (ytma) {
      if (bn == 128) return launch_pairs<128, false, true>(x16, s_x, M, K, lins, n_lin, raw_s32, pairs, stream, sync);
      if (bn == 192) return launch_pairs<192, false, true>(x16, s_x, M, K, lins, n_lin, raw_s32, pairs, stream, sync);
      return launch_pairs<256, false, true>(x16, s_x, M, K, lins, n_lin, raw_s32, pairs, stream, sync);
    }
    if (unscale) {
      if (bn == 128) return launch_pairs<128, true, false>(x16, s_x, M, K, lins, n_lin, raw_s32, pairs, stream, sync);
      if (bn == 192) return launch_pairs<192, true, false>(x16, s_x, M, K, lins, n_lin, raw_s32, pairs, stream, sync);
      return launch_pairs<256, true, false>(x16, s_x, M, K, lins, n_lin, raw_s32, pairs, stream, sync);
    }
    if (bn == 128) return launch_pairs<128, false, false>(x16, s_x, M, K, lins, n_lin, raw_s32, pairs, stream, sync);
    if (bn == 192) return launch_pairs<192, false, false>(x16, s_x, M, K, lins, n_lin, raw_s32, pairs, stream, sync);
    return launch_pairs<256, false, false>(x16, s_x, M, K, lins, n_lin, raw_s32, pairs, stream, sync);
  }
  GemmParams p;
  if (int st = fill_params<1, 256>(p, x16, s_x, M, K, lins, n_lin, raw_s32)) return st;
  if (p.total_tiles == 0) return CONVROT_OK;
  const int grid = std::min(p.total_tiles, device_sm_count());
  if (unscale) {
    if (int st = configure_kernel<1, 256, true, false>()) return st;
    convrot_gemm_kernel<1, 256, true, false><<<grid, THREADS, Geom<1, 256>::SMEM_ALLOC, stream>>>(p);
  } else {
    if (int st = configure_kernel<1, 256, false, false>()) return st;
    convrot_gemm_kernel<1, 256, false, false><<<grid, THREADS, Geom<1, 256>::SMEM_ALLOC, stream>>>(p);
  }
  return check_launch();
}

namespace {

// The epilogue's unscaling step (neg_unscale_f32x2) against the IEEE division
// for one divisor per blockIdx.y and every significand of y = 1.m * 2^y_exp,
// two at a time; counts the results that differ in any bit and keeps the
// smallest (divisor index, y bits) of those.
constexpr int SWEEP_THREADS = 256;
constexpr int SWEEP_PER_THREAD = 16;  // significands per thread, in pairs
__global__ void __launch_bounds__(SWEEP_THREADS) unscale_sweep_kernel(const float* __restrict__ divisors,
                                                                      int y_exp, unsigned long long* mismatches,
                                                                      unsigned long long* first) {
  const float a = divisors[blockIdx.y];
  const Unscale u = make_unscale(a);
  const uint32_t e_bits = static_cast<uint32_t>(y_exp + 127) << 23;
  const uint32_t m0 = (blockIdx.x * SWEEP_THREADS + threadIdx.x) * SWEEP_PER_THREAD;
  unsigned n_bad = 0;
  unsigned long long worst = ~0ull;
#pragma unroll
  for (int i = 0; i < SWEEP_PER_THREAD; i += 2) {
    const float y0 = __uint_as_float(e_bits | (m0 + i)), y1 = __uint_as_float(e_bits | (m0 + i + 1));
    float n0, n1;
    unpair_f32(neg_unscale_f32x2(pair_f32(y0, y1), u), n0, n1);
    const bool bad0 = __float_as_uint(-n0) != __float_as_uint(__fdiv_rn(y0, a));
    const bool bad1 = __float_as_uint(-n1) != __float_as_uint(__fdiv_rn(y1, a));
    const unsigned long long tag = static_cast<unsigned long long>(blockIdx.y) << 32;
    if (bad0) worst = min(worst, tag | __float_as_uint(y0));
    if (bad1) worst = min(worst, tag | __float_as_uint(y1));
    n_bad += bad0 + bad1;
  }
  if (n_bad) {
    atomicAdd(mismatches, static_cast<unsigned long long>(n_bad));
    atomicMin(first, worst);
  }
}

}  // namespace

int launch_unscale_sweep(const float* divisors, int n_divisors, int y_exp, unsigned long long* mismatches,
                         unsigned long long* first, cudaStream_t stream) {
  constexpr int per_block = SWEEP_THREADS * SWEEP_PER_THREAD;
  static_assert((1 << 23) % per_block == 0, "whole blocks of significands");
  const dim3 grid((1 << 23) / per_block, n_divisors);
  unscale_sweep_kernel<<<grid, SWEEP_THREADS, 0, stream>>>(divisors, y_exp, mismatches, first);
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
