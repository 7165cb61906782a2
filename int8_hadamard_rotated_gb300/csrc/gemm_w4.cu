// gemm_w4.cu -- the exact S8 x S4 GEMM of the packed INT4 convrot format,
// reading the weights in their checkpoint byte layout.
//
// What it computes (stable-diffusion.cpp docs, page "INT8 Convrot
// Safetensors", section "Packed INT4 convrot"): convrot_w4a4 weights are
// signed 4-bit values, low nibble first (element 2j of a row is the low
// nibble of byte j, element 2j+1 its high nibble), with an F32 per-output
// weight scale; the activations use the INT8 convrot pack. The product is
// A[r,o] = sum_i Q_x[r,i] Q_w[o,i] in int32, reconstructed like the INT8
// linear, Y = float(A) * s_x[r] * s_w[o] + b[o], one fp32 rounding per
// operation in that order; the packed weights are not expanded.
//
// Exactness. |Q_x| <= 127 and |Q_w| <= 8, so a run of K <= 16384 products
// keeps every partial sum below 127 * 8 * 16384 = 16,646,144 < 2^24: the fp32
// tensor-memory accumulator of a whole tile holds the exact integer A, and A
// itself is below 2^24, so float(A) is exact too. The launcher accepts
// K <= CONVROT_W4_MAX_K (16384) only.
//
// Kernel shape. Persistent CTA pairs (clusters of two, cta_group::2) on tiles
// of 256 weight rows x BN activation rows, like the binary16 kernel, with 19
// warps per CTA and three rings of shared-memory slots, each stepped once per
// 64-deep K block:
//   activation ring (6-8 slots): binary16 activation codes, loaded by the pair
//     TMA of warp 15 as soon as the MMAs release a slot;
//   packed ring (8 slots): the CTA's 128 rows of packed weight bytes (4 KB per
//     block), loaded by warp 8 up to 8 blocks ahead;
//   weight ring (4 slots): the binary16 weight tile (16 KB, 128-byte swizzle,
//     the layout a tensor-map load of binary16 codes would give), written by
//     the eight converter warps (9, 10, 12-14, 16-18) in four pairs. Pair q widens every block
//     whose index in the CTA's block stream is q modulo 4, each warp half of
//     its rows, so four blocks are in conversion at once and the latency of
//     each (its shared-memory stores must drain before the proxy fence lets
//     the tensor cores read them) overlaps the others.
//   warp 11     MMA issuer (the even CTA): once a block's activation slot is
//               full and both CTAs' converter warps have signalled its weight
//               slot, tcgen05.mma kind::f16 (M = 256, N = BN) into one of two
//               TMEM accumulators; the commits release both slots in both CTAs.
//   warps 0-7   epilogue: one accumulator column block of 32 rows at a time
//               from TMEM, reconstructed and stored through shared memory
//               with tensor-map stores (each thread owns one output feature).
// The converters of the odd CTA signal the even CTA's barrier with a
// CTA-scope release: the weight tile they wrote is in their own shared
// memory, read by their own SM's tensor cores after the proxy fence, so the
// signal only has to follow those writes (a cluster-scope release cost about
// 0.7 us per block and halved the throughput).
#include "gemm_common.cuh"

#include <algorithm>
#include <cstring>
#include <mutex>

namespace convrot {

// Sticky device error word of the S8 x S4 GEMM (timeouts of bounded waits).
__device__ int g_w4_error = 0;

namespace {

using namespace gemm;

constexpr int CONV_WARPS = 8;                     // four pairs, one K block per pair, round-robin
// Warp roles. Warp w issues on scheduler w mod 4. The MMA issuer paces the
// whole kernel, so it shares its scheduler only with light warps (two
// epilogue warps, which idle between tiles, and the activation loader); the
// converters' bursts of widening arithmetic run on the other three.
constexpr int W4_WARPS = NUM_EPI_WARPS + 3 + CONV_WARPS;  // 19
constexpr int W4_MMA_WARP = 11;        // scheduler 3
constexpr int X_PRODUCER_WARP = 15;    // scheduler 3
constexpr int PK_PRODUCER_WARP = 8;    // scheduler 0
constexpr int W4_THREADS = W4_WARPS * 32;
__host__ __device__ constexpr bool conv_slot(int w) {
  return w >= NUM_EPI_WARPS && w < W4_WARPS && w != W4_MMA_WARP && w != X_PRODUCER_WARP && w != PK_PRODUCER_WARP;
}
// Index of converter warp w among the converter warps (0 .. CONV_WARPS - 1).
__host__ __device__ constexpr int conv_index(int w) {
  int i = 0;
  for (int v = NUM_EPI_WARPS; v < w; ++v) i += conv_slot(v) ? 1 : 0;
  return i;
}
static_assert(conv_index(W4_WARPS) == CONV_WARPS, "every remaining warp converts");
static_assert((W4_MMA_WARP & 3) == (X_PRODUCER_WARP & 3) && (W4_MMA_WARP & 3) != (PK_PRODUCER_WARP & 3),
              "no converter shares the MMA warp's scheduler");
constexpr int PW_BYTES = CTA_M * BK / 2;  // packed weight bytes of one CTA per K block (4 KB)
constexpr int W4_TILE_M = 2 * CTA_M;
constexpr int CONV_PAIRS = CONV_WARPS / 2;  // pair q widens the blocks q (mod CONV_PAIRS)
constexpr int W_SLOTS = CONV_PAIRS;         // binary16 weight ring: slot q belongs to pair q
constexpr int PK_SLOTS = 2 * CONV_PAIRS;    // packed ring (prefetch depth): slots q, q + CONV_PAIRS for pair q
constexpr int DONE_SLOTS = 8;               // "block done" ring: one MMA commit per block

static_assert(127 * 8 * CONVROT_W4_MAX_K < (1 << 24), "one tile must stay exact in fp32");
static_assert(PW_BYTES % (2 * 32 * 16) == 0, "a converter warp widens whole 16-byte chunks per lane");
static_assert(W_SLOTS % CONV_PAIRS == 0 && PK_SLOTS % CONV_PAIRS == 0 && DONE_SLOTS % CONV_PAIRS == 0,
              "every slot is waited on by one converter pair only, in order");
static_assert((DONE_SLOTS & (DONE_SLOTS - 1)) == 0 && (CONV_PAIRS & (CONV_PAIRS - 1)) == 0 &&
                  (PK_SLOTS & (PK_SLOTS - 1)) == 0,
              "ring indices by masks");

template <int BN_>
struct GeomW4 {
  static constexpr int BN = BN_;
  static constexpr int COLS = BN / 2;          // columns (activation rows) per epilogue thread
  static constexpr int X_ROWS = BN / 2;        // activation rows each CTA loads
  static constexpr int W_BYTES = CTA_M * BK * 2;
  static constexpr int X_BYTES = X_ROWS * BK * 2;
  // fixed part: weight and packed rings, Y staging, row scales, barriers, misc, alignment slack
  static constexpr int FIXED = W_SLOTS * W_BYTES + PK_SLOTS * PW_BYTES + 2 * Y_HALF_BYTES + 2 * 128 * 4 + 1024 + 1024;
  static constexpr int X_RAW = (227 * 1024 - FIXED) / X_BYTES;
  static constexpr int X_SLOTS = X_RAW > 8 ? 8 : X_RAW;
  static constexpr uint32_t IDESC = idesc_f16_f32(W4_TILE_M, BN);
  // shared-memory layout (after aligning the base to 1024 B)
  static constexpr int SMEM_X = 0;                                     // [X_SLOTS][X_ROWS][64] binary16
  static constexpr int SMEM_W = X_SLOTS * X_BYTES;                     // [W_SLOTS][128][64] binary16
  static constexpr int SMEM_PW = SMEM_W + W_SLOTS * W_BYTES;           // [PK_SLOTS][128][32] packed bytes
  static constexpr int SMEM_YOUT = SMEM_PW + PK_SLOTS * PW_BYTES;      // [2][2][Y_ROWS][128] fp32
  static constexpr int SMEM_SX = SMEM_YOUT + 2 * Y_HALF_BYTES;         // [2][128] fp32 row scales
  static constexpr int SMEM_BARS = SMEM_SX + 2 * 128 * 4;
  // x_full [X]; w_full [W]; done [DONE]; pk_full, pk_empty [PK]; tfull, tempty [2]; drain
  static constexpr int NUM_BARS = X_SLOTS + W_SLOTS + DONE_SLOTS + 2 * PK_SLOTS + 2 + 2 + 1;
  static constexpr int SMEM_MISC = SMEM_BARS + NUM_BARS * 8;           // tmem base (u32), abort flag (int)
  static constexpr int SMEM_ALLOC = SMEM_MISC + 16 + 1024;
};
static_assert(GeomW4<256>::X_SLOTS >= 5 && GeomW4<256>::SMEM_ALLOC <= 227 * 1024 &&
                  GeomW4<192>::SMEM_ALLOC <= 227 * 1024 && GeomW4<128>::SMEM_ALLOC <= 227 * 1024,
              "shared memory");

// Arrive on the even CTA's mbarrier at shared::cluster address `addr` with a
// CTA-scope release (see the kernel description).
__device__ __forceinline__ void mbar_arrive_remote_cta(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}

// Eight signed 4-bit values (one 32-bit word of the packed row, element 2j in
// the low nibble of byte j) -> four binary16 pairs in element order. Pair k
// takes byte k into both halves (one byte permute); one LOP3 keeps the low
// nibble n0 in the low half and the high nibble n1 (at bits 4-7) in the high
// half and sets the bits 0x6400 | (n0 ^ 8) and 0x6400 | ((n1 ^ 8) << 4): the
// binary16 numbers 1024 + v0 + 8 and 1024 + 16 (v1 + 8) for the nibbles'
// two's-complement values v0, v1. One HFMA2, (x0, x1) * (1, 1/16) +
// (-1032, -72), gives (v0, v1): every product and sum is an integer below
// 2^11 or that divided by 16 exactly, so the fused operation is exact.
__device__ __forceinline__ void widen_w4x8(uint32_t w, uint32_t (&h)[4]) {
  const __half2 scale = __floats2half2_rn(1.0f, 0.0625f);
  const __half2 offset = __floats2half2_rn(-1032.0f, -72.0f);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t t = (__byte_perm(w, 0u, static_cast<uint32_t>(k | (k << 8))) & 0x00F0000Fu) ^ 0x64806408u;
    __half2 v = __hfma2(*reinterpret_cast<const __half2*>(&t), scale, offset);
    h[k] = *reinterpret_cast<uint32_t*>(&v);
  }
}

// GELU: the output is gelu(y) (gelu_as2: the Abramowitz & Stegun 7.1.28 erf;
// the MLP's activation applied where the up linear's output is stored).
template <int BN_, bool UNSCALE, bool GELU = false>
__global__ void __launch_bounds__(W4_THREADS, 1)
convrot_gemm_w4_kernel(const __grid_constant__ GemmParams p) {
  using Gm = GeomW4<BN_>;
  constexpr int BN = Gm::BN;
  constexpr int COLS = Gm::COLS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  constexpr int XS = Gm::X_SLOTS;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Gm::SMEM_BARS);
  uint64_t* x_full = bars;                          // [XS] (even CTA: both CTAs' activation bytes)
  uint64_t* w_full = x_full + XS;                   // [W_SLOTS] (even CTA: the converter pairs of both CTAs)
  uint64_t* done = w_full + W_SLOTS;                // [DONE_SLOTS] the pair's MMAs of block n finished (n mod 8)
  uint64_t* pk_full = done + DONE_SLOTS;            // [PK_SLOTS] this CTA's packed bytes landed
  uint64_t* pk_empty = pk_full + PK_SLOTS;          // [PK_SLOTS] this CTA's converter read them
  uint64_t* tfull = pk_empty + PK_SLOTS;            // [2]
  uint64_t* tempty = tfull + 2;                     // [2]
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(smem + Gm::SMEM_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Gm::SMEM_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int* err = &g_w4_error;
  const uint32_t rank = cluster_ctarank();  // 0: the pair's leader (issues the MMAs)
  const bool leader = (rank == 0);
  const int unit = static_cast<int>(cluster_id_x());
  const int n_units = static_cast<int>(cluster_count_x());
  constexpr uint16_t pair_mask = 0x3u;

  if (threadIdx.x == X_PRODUCER_WARP * 32) {
    for (int s = 0; s < XS; ++s) mbar_init(&x_full[s], 1);
    for (int s = 0; s < W_SLOTS; ++s) mbar_init(&w_full[s], 4);  // the two warps of a converter pair in each CTA
    for (int s = 0; s < DONE_SLOTS; ++s) mbar_init(&done[s], 1);
    for (int s = 0; s < PK_SLOTS; ++s) {
      mbar_init(&pk_full[s], 1);
      mbar_init(&pk_empty[s], 2);  // the two warps of this CTA's converter pair
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], NUM_EPI_WARPS * 2);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&p.tmap_x);
    for (int j = 0; j < p.n_lin; ++j) tma_prefetch_desc(&p.tmap_w[j]);
  }
  if (warp == W4_MMA_WARP) {
    tmem_alloc_pair(tmem_base_smem, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_smem;
  // launched as a programmatic dependent of the kernel before it (the pack):
  // no global memory is touched before that kernel has completed
  pdl_wait_prerequisites();

  if (warp == X_PRODUCER_WARP || warp == PK_PRODUCER_WARP) {
    // the two loaders: activation blocks into the activation ring (pair TMA,
    // completing on the even CTA's barrier), packed weight blocks into the
    // packed ring (this CTA's barrier)
    if (lane == 0) {
      const bool is_x = (warp == X_PRODUCER_WARP);
      const uint64_t pol = l2_policy_evict_normal();
      const uint32_t x_full_leader = mapa_shared(smem_u32(x_full), 0);
      const uint32_t slots = is_x ? XS : PK_SLOTS;
      uint32_t n = 0;           // block index in this CTA's stream
      uint32_t s = 0, ph = 0;   // its slot and the slot's use parity
      bool ok = true;
      WorkItem it;
      for (int j = 0; ok && work_item(p, unit, n_units, j, it); ++j) {
        const TileCoord c = decode_tile(p, it.t);
        const int w_row = c.wt * W4_TILE_M + static_cast<int>(rank) * CTA_M;
        const int x_row = c.xt * BN + static_cast<int>(rank) * Gm::X_ROWS;
        for (int kb = it.kb0; kb < it.kb1; ++kb, ++n) {
          if (is_x) {
            // the slot is free once the MMAs of block n - XS have finished
            if (n >= slots) {
              const uint32_t m = n - slots;
              if (!mbar_wait(&done[m & (DONE_SLOTS - 1)], (m / DONE_SLOTS) & 1u, abort_flag, err, p.wait_ns)) { ok = false; break; }
            }
            if (leader) mbar_arrive_expect_tx(&x_full[s], 2 * Gm::X_BYTES);
            tma_load_2d_pair(smem + Gm::SMEM_X + s * Gm::X_BYTES, &p.tmap_x, x_full_leader + s * 8u, kb * BK,
                             x_row, pol);
          } else {
            if (!mbar_wait(&pk_empty[s], ph ^ 1u, abort_flag, err, p.wait_ns)) { ok = false; break; }
            mbar_arrive_expect_tx(&pk_full[s], PW_BYTES);
            tma_load_2d(smem + Gm::SMEM_PW + s * PW_BYTES, &p.tmap_w[c.lin], &pk_full[s], kb * (BK / 2), w_row,
                        pol);
          }
          if (++s == slots) { s = 0; ph ^= 1u; }
        }
      }
      // no copy may land after the CTAs exit: wait (bounded) for the last
      // phase of every slot that was filled
      for (uint32_t t = 0; t < slots; ++t)
        if (n > t) {
          const uint32_t tph = ((n - 1 - t) / slots) & 1u;
          if (!is_x) mbar_wait(&pk_full[t], tph, nullptr, err, p.wait_ns);
          else if (leader) mbar_wait(&x_full[t], tph, nullptr, err, p.wait_ns);
        }
    }
    __syncwarp();
  } else if (warp == W4_MMA_WARP) {
    if (lane == 0 && leader) {
      uint32_t acc_iter = 0;
      uint32_t xs = 0, xph = 0, ws = 0, wph = 0, ds = 0;  // ring positions of the next block
      const uint64_t a_desc0 = smem_desc_sw128(smem_u32(smem + Gm::SMEM_W));
      const uint64_t b_desc0 = smem_desc_sw128(smem_u32(smem + Gm::SMEM_X));
      bool ok = true;
      WorkItem it;
      for (int j = 0; ok && work_item(p, unit, n_units, j, it); ++j) {
        const uint32_t buf = acc_iter & 1u;
        const uint32_t use = acc_iter >> 1;
        if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort_flag, err, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        for (int kb = it.kb0; kb < it.kb1; ++kb) {
          if (!mbar_wait(&x_full[xs], xph, abort_flag, err, p.wait_ns)) { ok = false; break; }
          if (!mbar_wait(&w_full[ws], wph, abort_flag, err, p.wait_ns)) { ok = false; break; }
          tc_fence_after();
          // descriptors advance by the slot offset (address >> 4 in the low field)
          const uint64_t a_desc = a_desc0 + static_cast<uint64_t>(ws * (Gm::W_BYTES >> 4));
          const uint64_t b_desc = b_desc0 + static_cast<uint64_t>(xs * (Gm::X_BYTES >> 4));
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            const uint64_t koff = static_cast<uint64_t>((k * UMMA_K * 2) >> 4);
            mma_f16_ss_pair(d_tmem, a_desc + koff, b_desc + koff, Gm::IDESC, (kb > it.kb0 || k > 0) ? 1u : 0u);
          }
          mma_commit_pair(&done[ds], pair_mask);
          if (++xs == static_cast<uint32_t>(XS)) { xs = 0; xph ^= 1u; }
          if (++ws == static_cast<uint32_t>(W_SLOTS)) { ws = 0; wph ^= 1u; }
          ds = (ds + 1) & (DONE_SLOTS - 1);
        }
        if (!ok) break;
        mma_commit_pair(&tfull[buf], pair_mask);
        ++acc_iter;
      }
      // all issued MMAs complete before TMEM is released
      mma_commit_pair(drain, 0x1u);
      mbar_wait(drain, 0, nullptr, err, p.wait_ns);
    }
    __syncwarp();
  } else if (conv_slot(warp)) {
    // ---------------------------- converters -------------------------------
    // Converter pair q (warps q and q + CONV_PAIRS) widens the blocks
    // n = q (mod CONV_PAIRS) of this CTA's stream, always into weight slot q,
    // so each slot's barriers are waited on in order by one pair (a second
    // pair could see a phase two uses old as complete). Warp half hr of the
    // pair writes weight rows 64 hr .. +63: its lane l widens the 16-byte
    // chunks c = 128 hr + l + 32 i (i < 4) of the staged block. Chunk c holds
    // elements 32 (c & 1) .. +31 of weight row c >> 1, which become the row's
    // binary16 chunks 4 (c & 1) .. +3 (8 elements each) at their
    // 128-byte-swizzle positions.
    const int cw = conv_index(warp);
    const uint32_t q = static_cast<uint32_t>(cw % CONV_PAIRS);
    const int hr = cw / CONV_PAIRS;
    const uint32_t w_full_leader = mapa_shared(smem_u32(w_full), 0);
    uint32_t n = 0;
    bool ok = true;
    WorkItem it;
    for (int j = 0; ok && work_item(p, unit, n_units, j, it); ++j) {
      for (int kb = it.kb0; kb < it.kb1; ++kb, ++n) {
        if ((n & (CONV_PAIRS - 1)) != q) continue;
        const uint32_t ps = n & (PK_SLOTS - 1), ws = n % W_SLOTS;
        if (!mbar_wait(&pk_full[ps], (n / PK_SLOTS) & 1u, abort_flag, err, p.wait_ns)) { ok = false; break; }
        // widen into registers first (off the weight slot's critical path),
        // hand the packed slot back, then store once the weight slot is free
        constexpr int NCH = PW_BYTES / (2 * 32 * 16);  // 16-byte chunks per lane
        const uint8_t* spw = smem + Gm::SMEM_PW + ps * PW_BYTES;
        uint32_t h[NCH][16];
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
          const int c = (PW_BYTES / 32) * hr + lane + 32 * i;
          const uint4 in = *reinterpret_cast<const uint4*>(spw + 16 * c);
          widen_w4x8(in.x, *reinterpret_cast<uint32_t(*)[4]>(&h[i][0]));
          widen_w4x8(in.y, *reinterpret_cast<uint32_t(*)[4]>(&h[i][4]));
          widen_w4x8(in.z, *reinterpret_cast<uint32_t(*)[4]>(&h[i][8]));
          widen_w4x8(in.w, *reinterpret_cast<uint32_t(*)[4]>(&h[i][12]));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&pk_empty[ps]);  // the packed bytes are in registers: reload the slot
        // the weight slot is free once the MMAs of block n - W_SLOTS have finished
        if (n >= static_cast<uint32_t>(W_SLOTS)) {
          const uint32_t m = n - W_SLOTS;
          if (!mbar_wait(&done[m & (DONE_SLOTS - 1)], (m / DONE_SLOTS) & 1u, abort_flag, err, p.wait_ns)) { ok = false; break; }
        }
        uint8_t* sw = smem + Gm::SMEM_W + ws * Gm::W_BYTES;
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
          const int c = (PW_BYTES / 32) * hr + lane + 32 * i;
          const int r = c >> 1, hpart = c & 1;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const int chunk = (4 * hpart + m) ^ (r & 7);
            *reinterpret_cast<uint4*>(sw + r * 128 + chunk * 16) =
                make_uint4(h[i][4 * m], h[i][4 * m + 1], h[i][4 * m + 2], h[i][4 * m + 3]);
          }
        }
        fence_proxy_async_smem();  // the tensor cores read this tile through the async proxy
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(&w_full[ws]);
          else mbar_arrive_remote_cta(w_full_leader + ws * 8u);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------ epilogue ------------------------------
    const int quarter = warp & 3;             // TMEM lanes 32*quarter .. +31
    const int half = warp >> 2;               // activation columns half*COLS .. +COLS-1
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    const uint32_t tempty_leader = mapa_shared(smem_u32(tempty), 0);
    const uint64_t pol_y = l2_policy_evict_first();
    uint32_t acc_iter = 0;
    WorkItem it;
    for (int j = 0; work_item(p, unit, n_units, j, it); ++j) {
      const TileCoord c = decode_tile(p, it.t);
      const int N = p.N[c.lin];
      const int o = c.wt * W4_TILE_M + static_cast<int>(rank) * CTA_M + 32 * quarter + lane;
      const bool o_ok = o < N;
      const int r0 = c.xt * BN + half * COLS;
      int32_t* part = static_cast<int32_t*>(p.out[c.lin]);  // partial sums of a split tile, as int32
      bool ok = true;
      if (it.kind == kTail) {
        if (threadIdx.x == 0) {
          unsigned long long* f = p.sk_flags + 2 * (unit - 1) + rank;
          ok = wait_flag(f, p.epoch ^ p.handover_xor, abort_flag, err, p.wait_ns);
          if (ok) st_relaxed_gpu(f, 0ull);  // consumed: zero again for the next launch
        }
      }
      const uint32_t buf = acc_iter & 1u;
      const uint32_t use = acc_iter >> 1;
      if (ok) ok = mbar_wait(&tfull[buf], use & 1u, abort_flag, err, p.wait_ns);
      // the eight epilogue warps agree before any barrier of the stores below
      if (!named_bar_and(EPI_BAR, NUM_EPI_WARPS * 32, ok)) break;
      tc_fence_after();
      const float* sw_ptr = p.s_w[c.lin];
      const float* b_ptr = p.bias[c.lin];
      const float sw = (o_ok && sw_ptr) ? __ldg(sw_ptr + o) : 1.0f;
      const float bb = (o_ok && b_ptr) ? __ldg(b_ptr + o) : 0.0f;
      const float in_scale = UNSCALE ? p.in_scale[c.lin] : 1.0f;
      const unsigned long long sw2 = pair_f32(sw, sw), bb2 = pair_f32(bb, bb);
      uint8_t* sy_base = smem + Gm::SMEM_YOUT + half * Y_HALF_BYTES;
      const bool store_leader = (quarter == 0 && lane == 0);
      const int col = 32 * quarter + lane;
      const int o_base = c.wt * W4_TILE_M + static_cast<int>(rank) * CTA_M;
      float* ssx = reinterpret_cast<float*>(smem + Gm::SMEM_SX) + half * 128;
      const bool staged = !p.raw_s32 && it.kind != kHead;
      if (staged && col < COLS) ssx[col] = (r0 + col < p.M) ? __ldg(p.s_x + r0 + col) : 0.0f;
      // unscaling: the tile's extreme row scales decide, per thread, whether
      // the correction step may replace the division
      Unscale us{};
      bool us_fast = false;
      if (UNSCALE && staged) {
        named_bar_sync(1 + half, 4 * 32);
        float v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = (lane + 32 * k < COLS) ? ssx[lane + 32 * k] : 0.0f;
        float lo, hi;
        warp_scale_range(v, lo, hi);
        us = make_unscale(in_scale);
        us_fast = unscale_fast_ok(in_scale, lo, hi, sw);
      }
      const unsigned long long m1 = pair_f32(-1.0f, -1.0f);
#pragma unroll 1
      for (int q = 0; q < COLS / 32; ++q) {
        uint32_t acc[32];
        tmem_ld_32x32b_x32(tmem_base + lane_base + buf * BN + half * COLS + q * 32, acc);
        tmem_ld_wait();
        if (q == COLS / 32 - 1) {
          // the accumulator is in registers: release it to the MMA
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(tempty_leader + buf * 8u);
        }
        const int rq = r0 + 32 * q;
        if (it.kind == kHead) {
          if (o_ok) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (rq + i < p.M) part[static_cast<int64_t>(rq + i) * N + o] = __float2int_rz(__uint_as_float(acc[i]));
          }
          continue;
        }
        if (it.kind == kTail && o_ok) {
          // the other pair's int32 partial sums (L2 loads: written by another SM)
#pragma unroll
          for (int i0 = 0; i0 < 32; i0 += 16) {
            int32_t v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = (rq + i0 + i < p.M) ? __ldcg(part + static_cast<int64_t>(rq + i0 + i) * N + o) : 0;
#pragma unroll
            for (int i = 0; i < 16; ++i)
              acc[i0 + i] = __float_as_uint(__int2float_rn(__float2int_rz(__uint_as_float(acc[i0 + i])) + v[i]));
          }
        }
        // acc now holds float(A) (|A| < 2^24: exact)
        if (p.raw_s32) {
          if (o_ok) {
            int32_t* A = static_cast<int32_t*>(p.out[c.lin]);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (rq + i < p.M) st_global_hint(A + static_cast<int64_t>(rq + i) * N + o,
                                               __float2int_rz(__uint_as_float(acc[i])), pol_y);
          }
          continue;
        }
#pragma unroll
        for (int sq = 0; sq < 32 / Y_ROWS; ++sq) {
          const int sub = q * (32 / Y_ROWS) + sq;  // block of Y_ROWS rows within the tile
          // every block commits one bulk group and a tile stores an even
          // number of blocks, so the group two back is the last store from
          // this buffer: wait until it has read it
          float* sy = reinterpret_cast<float*>(sy_base + (sub & 1) * Y_BUF_BYTES);
          if (store_leader) bulk_wait_read<1>();
          named_bar_sync(1 + half, 4 * 32);
#pragma unroll
          for (int i = 0; i < Y_ROWS; i += 4) {
            const int idx = sub * Y_ROWS + i;   // row within this warpgroup's COLS
            const int ai = sq * Y_ROWS + i;     // index into acc
            const float4 s4 = *reinterpret_cast<const float4*>(ssx + idx);
            // float(A) * s_x * s_w (/ input scale) + b, one rounding per operation, in that order
            unsigned long long ya = mul_f32x2(pair_f32(__uint_as_float(acc[ai]), __uint_as_float(acc[ai + 1])),
                                              pair_f32(s4.x, s4.y));
            unsigned long long yb = mul_f32x2(pair_f32(__uint_as_float(acc[ai + 2]), __uint_as_float(acc[ai + 3])),
                                              pair_f32(s4.z, s4.w));
            if (sw_ptr) {
              ya = mul_f32x2(ya, sw2);
              yb = mul_f32x2(yb, sw2);
            }
            if (UNSCALE && us_fast) {
              // -RN(y / a) by the correction step, then RN(b - (-q)) or -(-q)
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
              if (UNSCALE) {
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
            if (GELU) {
              gelu_as2(y0, y1);
              gelu_as2(y2, y3);
            }
            sy[i * CTA_M + col] = y0;
            sy[(i + 1) * CTA_M + col] = y1;
            sy[(i + 2) * CTA_M + col] = y2;
            sy[(i + 3) * CTA_M + col] = y3;
          }
          fence_proxy_async_smem();
          named_bar_sync(1 + half, 4 * 32);
          if (store_leader) {
            if (o_base < N && r0 + sub * Y_ROWS < p.M) tma_store_2d(&p.tmap_y[c.lin], sy, o_base, r0 + sub * Y_ROWS);
            bulk_commit();
          }
        }
      }
      if (it.kind == kHead) {
        // publish the partial sums to the pair that finishes the tile
        __threadfence();
        named_bar_sync(EPI_BAR, NUM_EPI_WARPS * 32);
        if (threadIdx.x == 0) st_release_gpu(p.sk_flags + 2 * unit + rank, p.epoch);
      }
      ++acc_iter;
    }
    // the last tensor-map stores complete before the CTA releases its shared memory
    if ((warp & 3) == 0 && lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  cluster_sync();
  if (warp == W4_MMA_WARP) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// Packed 4-bit weights [rows, K/2] bytes, box 32 bytes (64 values) x 128 rows,
// no swizzle, zero fill past the last row.
int make_tmap_w4(CUtensorMap* m, const void* base, int64_t rows, int64_t K) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return set_cuda_error(cudaErrorNotSupported);
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK / 2), static_cast<cuuint32_t>(CTA_M)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_cuda_error(cudaErrorInvalidValue);
  return CONVROT_OK;
}

template <int BN>
int fill_params_w4(GemmParams& p, const __half* x16, const float* s_x, int64_t M, int64_t K,
                   const GemmLinear* lins, int n_lin, bool raw_s32) {
  memset(&p, 0, sizeof(p));
  if (int st = make_tmap(&p.tmap_x, x16, M, K, BN / 2)) return st;
  int wt = 0;
  for (int j = 0; j < n_lin; ++j) {
    if (int st = make_tmap_w4(&p.tmap_w[j], lins[j].w4, lins[j].N, K)) return st;
    if (!raw_s32)
      if (int st = make_tmap_y(&p.tmap_y[j], lins[j].out, M, lins[j].N, CTA_M)) return st;
    p.s_w[j] = lins[j].s_w;
    p.bias[j] = lins[j].bias;
    p.kchunk[j] = nullptr;
    p.in_scale[j] = lins[j].in_scale;
    p.out[j] = lins[j].out;
    p.N[j] = static_cast<int>(lins[j].N);
    p.wtile_start[j] = wt;
    wt += static_cast<int>((lins[j].N + W4_TILE_M - 1) / W4_TILE_M);
  }
  p.wtile_start[n_lin] = wt;
  p.s_x = s_x;
  p.M = static_cast<int>(M);
  p.K = static_cast<int>(K);
  p.num_kb = static_cast<int>(K / BK);
  p.n_xtiles = static_cast<int>((M + BN - 1) / BN);
  p.n_wtiles = wt;
  const int64_t band_bytes = static_cast<int64_t>(BN) * K * 2;
  p.raster_bands = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(p.n_xtiles, RASTER_L2_BYTES / band_bytes)));
  const int64_t total = static_cast<int64_t>(p.n_xtiles) * wt;
  if (total > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
  p.total_tiles = static_cast<int>(total);
  p.n_lin = n_lin;
  p.raw_s32 = raw_s32 ? 1 : 0;
  p.wait_ns = kWaitLimitNs;
  p.handover_xor = 0;
  return CONVROT_OK;
}

template <int BN, bool UNSCALE, bool GELU = false>
int configure_w4() {
  static std::mutex mu;
  static uint64_t configured = 0;  // bit d: attribute set on device d
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_cuda_error(e);
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 64 || !((configured >> dev) & 1u)) {
    e = cudaFuncSetAttribute(convrot_gemm_w4_kernel<BN, UNSCALE, GELU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             GeomW4<BN>::SMEM_ALLOC);
    if (e != cudaSuccess) return set_cuda_error(e);
    if (dev < 64) configured |= (1ull << dev);
  }
  return CONVROT_OK;
}

// Co-resident CTA pairs of the BN variant (0 if they cannot launch), cached per device.
template <int BN>
int max_pairs_w4() {
  static std::mutex mu;
  static int cached[64];
  static bool known[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!known[dev]) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pair_config(device_sm_count() / 2, GeomW4<BN>::SMEM_ALLOC, nullptr, attr, false);
    cfg.blockDim = dim3(W4_THREADS, 1, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, convrot_gemm_w4_kernel<BN, false>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cached[dev] = n;
    known[dev] = true;
  }
  return cached[dev];
}

template <int BN, bool UNSCALE, bool GELU = false>
int launch_w4(const __half* x16, const float* s_x, int64_t M, int64_t K, const GemmLinear* lins, int n_lin,
              bool raw_s32, int pairs, cudaStream_t stream, const GemmSync& sync) {
  GemmParams p;
  if (int st = fill_params_w4<BN>(p, x16, s_x, M, K, lins, n_lin, raw_s32)) return st;
  if (p.total_tiles == 0) return CONVROT_OK;
  const int units = std::min(p.total_tiles, pairs);
  if (BN == 256) plan_split(p, units, 2, sync);
  if (int st = configure_w4<BN, UNSCALE, GELU>()) return st;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_config(units, GeomW4<BN>::SMEM_ALLOC, stream, attr, true);
  cfg.blockDim = dim3(W4_THREADS, 1, 1);
  cudaError_t e = cudaLaunchKernelEx(&cfg, convrot_gemm_w4_kernel<BN, UNSCALE, GELU>, p);
  if (e != cudaSuccess) return set_cuda_error(e);
  return check_launch();
}

}  // namespace

int launch_gemm_w4(const __half* x16, const float* s_x, int64_t M, int64_t K, const GemmLinear* lins, int n_lin,
                   bool raw_s32, cudaStream_t stream, GemmSync sync, bool gelu) {
  if (M == 0) return CONVROT_OK;
  if (K % 64 != 0 || K > CONVROT_W4_MAX_K) return CONVROT_ERR_UNSUPPORTED;
  bool unscale = false;
  for (int j = 0; j < n_lin; ++j) {
    unscale |= (lins[j].in_scale != 1.0f);
    if (!raw_s32 && lins[j].N % 4 != 0) return CONVROT_ERR_ALIGN;  // Y rows of whole 16-byte units
  }
  if (raw_s32 && unscale) return CONVROT_ERR_ARG;
  if (gelu && (raw_s32 || unscale)) return CONVROT_ERR_ARG;
  if (int st = configure_w4<256, false>()) return st;
  if (int st = configure_w4<192, false>()) return st;
  if (int st = configure_w4<128, false>()) return st;
  const int pairs = std::min(max_pairs_w4<256>(), std::min(max_pairs_w4<192>(), max_pairs_w4<128>()));
  if (pairs <= 0) return CONVROT_ERR_UNSUPPORTED;
  const bool can_split = sync.words && sync.bytes >= static_cast<size_t>(2 * pairs) * sizeof(unsigned long long);
  const int bn = pick_tile_rows(M, lins, n_lin, pairs, can_split);
  if (gelu) {
    if (bn == 128) return launch_w4<128, false, true>(x16, s_x, M, K, lins, n_lin, false, pairs, stream, sync);
    if (bn == 192) return launch_w4<192, false, true>(x16, s_x, M, K, lins, n_lin, false, pairs, stream, sync);
    return launch_w4<256, false, true>(x16, s_x, M, K, lins, n_lin, false, pairs, stream, sync);
  }
  if (unscale) {
    if (bn == 128) return launch_w4<128, true>(x16, s_x, M, K, lins, n_lin, raw_s32, pairs, stream, sync);
    if (bn == 192) return launch_w4<192, true>(x16, s_x, M, K, lins, n_lin, raw_s32, pairs, stream, sync);
    return launch_w4<256, true>(x16, s_x, M, K, lins, n_lin, raw_s32, pairs, stream, sync);
  }
  if (bn == 128) return launch_w4<128, false>(x16, s_x, M, K, lins, n_lin, raw_s32, pairs, stream, sync);
  if (bn == 192) return launch_w4<192, false>(x16, s_x, M, K, lins, n_lin, raw_s32, pairs, stream, sync);
  return launch_w4<256, false>(x16, s_x, M, K, lins, n_lin, raw_s32, pairs, stream, sync);
}

int read_and_clear_w4_error() {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_w4_error, sizeof(int));
  if (e != cudaSuccess) return set_cuda_error(e);
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_w4_error, &zero, sizeof(int));
    if (e != cudaSuccess) return set_cuda_error(e);
  }
  return v;
}

}  // namespace convrot
