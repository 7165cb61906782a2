// gemm_common.cuh -- definitions shared by the tensor-core GEMM kernels
// (gemm.cu: binary16 weight codes; gemm_w4.cu: packed 4-bit weight codes):
// tile geometry, the launch parameters, the split-wave work assignment, the
// raster order and the host-side helpers that build tensor maps and plan
// the split.
#pragma once

#include "common.cuh"

namespace convrot {
namespace gemm {

constexpr int BK = 64;                // K per pipeline stage: 64 fp16 = 128 B
constexpr int KB_PER_CHUNK = 16;      // 16 x 64 = 1024 products per exact chunk
constexpr int UMMA_K = 16;            // K of one kind::f16 MMA
constexpr int CTA_M = 128;            // weight rows per CTA (its TMEM lanes)
constexpr int NUM_EPI_WARPS = 8;
constexpr int PRODUCER_WARP = NUM_EPI_WARPS;
constexpr int MMA_WARP = NUM_EPI_WARPS + 1;
constexpr int THREADS = (NUM_EPI_WARPS + 2) * 32;
constexpr int TMEM_COLS = 512;       // two fp32 accumulators of BN columns each
constexpr int MAX_LIN = CONVROT_MAX_LINEARS;
constexpr int64_t RASTER_L2_BYTES = 48ll << 20;  // activation codes a raster group keeps in L2
constexpr int EPI_BAR = 3;            // named barrier of the eight epilogue warps (1, 2: per warpgroup)

static_assert(TMEM_COLS <= 512, "TMEM has 512 columns");
static_assert(KB_PER_CHUNK * BK * 127 * 127 < (1 << 24), "chunk must stay exact in fp32");

// Y staging for tensor-map stores: per epilogue warpgroup one buffer of
// Y_ROWS activation rows x 128 output features (fp32), two buffers per
// epilogue warpgroup used in turn, so that filling one overlaps the store of
// the other.
constexpr int Y_ROWS = 8;
constexpr int Y_BUF_BYTES = Y_ROWS * CTA_M * 4;
constexpr int Y_HALF_BYTES = 2 * Y_BUF_BYTES;  // one warpgroup's two buffers

template <int CG, int BN_, bool YTMA = false>
struct Geom {
  static constexpr int BN = BN_;                      // activation rows per tile (MMA N)
  static constexpr int COLS = BN / 2;                 // columns per epilogue thread (two warpgroups)
  static constexpr int TILE_M = CTA_M * CG;           // weight rows per tile (MMA M)
  static constexpr int X_ROWS = BN / CG;              // activation rows each CTA loads
  static constexpr int W_BYTES = CTA_M * BK * 2;
  static constexpr int X_BYTES = X_ROWS * BK * 2;
  static constexpr int STAGE_BYTES = W_BYTES + X_BYTES;
  static constexpr int STAGES = (196 * 1024) / STAGE_BYTES;  // 4 (CG 1), 6-8 (pairs)
  static constexpr uint32_t IDESC = idesc_f16_f32(TILE_M, BN);
  // shared-memory layout (after aligning the base to 1024 B)
  static constexpr int SMEM_YOUT = STAGES * STAGE_BYTES;                  // [2][2][Y_ROWS][128] fp32 (YTMA)
  static constexpr int SMEM_SX = SMEM_YOUT + (YTMA ? 2 * Y_HALF_BYTES : 0);  // [2][128] fp32 row scales (YTMA)
  static constexpr int SMEM_BARS = SMEM_SX + (YTMA ? 2 * 128 * 4 : 0);  // full[S], empty[S], tfull[2], tempty[2], drain
  static constexpr int NUM_BARS = 2 * STAGES + 2 + 2 + 1;
  static constexpr int SMEM_MISC = SMEM_BARS + NUM_BARS * 8;  // tmem base (u32), abort flag (int)
  // slack for the 1024-B alignment, and (pairs) one more half tile so that
  // every operand read of the last stage stays inside the allocation
  static constexpr int SMEM_ALLOC = SMEM_MISC + 16 + 1024;
};
static_assert(Geom<1, 256>::SMEM_ALLOC <= 227 * 1024 && Geom<2, 256, true>::SMEM_ALLOC <= 227 * 1024 &&
                  Geom<2, 192, true>::SMEM_ALLOC <= 227 * 1024 && Geom<2, 128, true>::SMEM_ALLOC <= 227 * 1024,
              "shared memory");
static_assert(2 * 256 <= TMEM_COLS, "two accumulators fit in TMEM");
static_assert((256 / 2 / Y_ROWS) % 2 == 0 && (192 / 2 / Y_ROWS) % 2 == 0 && (128 / 2 / Y_ROWS) % 2 == 0,
              "every tile height stores an even number of Y blocks per warpgroup");

struct GemmParams {
  CUtensorMap tmap_x;              // activation codes, fp16 [M, K], box X_ROWS x 64
  CUtensorMap tmap_w[MAX_LIN];     // weight codes, fp16 [N_j, K], box 128 x 64
  CUtensorMap tmap_y[MAX_LIN];     // fp32 Y_j [M, N_j], box 128 x Y_ROWS (YTMA kernels)
  const float* s_w[MAX_LIN];
  const float* bias[MAX_LIN];
  const int32_t* kchunk[MAX_LIN];  // exact-chunk plan per 128 weight rows, or null
  float in_scale[MAX_LIN];         // input scale to divide out before the bias (1 = none)
  void* out[MAX_LIN];              // fp32 Y_j or int32 A_j, [M, N_j]
  int N[MAX_LIN];
  int wtile_start[MAX_LIN + 1];    // prefix sums of weight tiles (TILE_M rows) per linear
  const float* s_x;
  int M;
  int K;
  int num_kb;                      // ceil(K / BK)
  int n_xtiles;                    // ceil(M / BN) activation bands
  int n_wtiles;                    // sum over linears of ceil(N_j / TILE_M)
  int total_tiles;                 // n_xtiles * n_wtiles
  int raster_bands;                // bands per raster group
  int n_lin;
  int raw_s32;
  // Balanced waves: the K blocks of the first sk_tiles tiles (0 = none) are
  // split into one contiguous range per unit, done first; the other tiles are
  // then taken whole, round-robin over the units. A unit whose range ends
  // inside a tile stores its int32 partial sums in that tile's output and
  // publishes `epoch` in its flag word; the unit whose range finishes the
  // tile adds them. Split tiles come first so that this hand-over overlaps
  // the whole tiles' MMAs instead of lengthening the last wave.
  int sk_tiles;
  unsigned long long* sk_flags;    // [2 * units]: one word per CTA of a pair
  unsigned long long epoch;        // nonzero, distinct per launch
  // Bounded waits: every wait of the launch gives up after wait_ns
  // (kWaitLimitNs normally). A test of the timeout path shortens it and sets
  // handover_xor, so that the tails of split tiles wait for epoch ^ handover_xor,
  // a value no head publishes (0 normally).
  unsigned long long wait_ns;
  unsigned long long handover_xor;
};

struct TileCoord {
  int lin, wt, xt;
};

// One piece of a unit's work: K blocks [kb0, kb1) of tile t.
enum : int {
  kWhole = 0,  // the whole tile
  kHead = 1,   // the tile's first K blocks: partial sums go to the next unit
  kTail = 2,   // the tile's last K blocks: adds the previous unit's partial sums
};
struct WorkItem {
  int t, kb0, kb1, kind;
};

// Item j of a unit's work: first its K-block range of the split tiles, from
// the highest tile down, so that the head it hands on comes first and the
// tail it finishes last; then its whole tiles. Every range is at least one
// tile long (sk_tiles >= units), so a split tile has exactly one head and one
// tail, and the tail's unit is the head's plus one. Items are recomputed from
// j rather than carried, to keep the epilogue's registers for its
// accumulators.
__device__ __forceinline__ bool work_item(const GemmParams& p, int unit, int n_units, int j, WorkItem& it) {
  int n_sk = 0;
  if (p.sk_tiles > 0) {
    const long long total = static_cast<long long>(p.sk_tiles) * p.num_kb;
    const int s = static_cast<int>(total * unit / n_units);
    const int e = static_cast<int>(total * (unit + 1) / n_units);
    const int hi = (e - 1) / p.num_kb;
    n_sk = hi - s / p.num_kb + 1;
    if (j < n_sk) {
      const int tile = hi - j;
      const int base = tile * p.num_kb;
      it.t = tile;
      it.kb0 = max(0, s - base);
      it.kb1 = min(p.num_kb, e - base);
      it.kind = (it.kb1 < p.num_kb) ? kHead : (it.kb0 > 0 ? kTail : kWhole);
      return true;
    }
  }
  const int t = p.sk_tiles + unit + (j - n_sk) * n_units;
  if (t >= p.total_tiles) return false;
  it.t = t;
  it.kb0 = 0;
  it.kb1 = p.num_kb;
  it.kind = kWhole;
  return true;
}

// Lane-wise IEEE fp32 pairs (each lane rounded as the scalar operation).
__device__ __forceinline__ unsigned long long pair_f32(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpair_f32(unsigned long long r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long mul_f32x2(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long add_f32x2(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Unscaling by a linear's input scale a (y / a, correctly rounded) without a
// division per element: Markstein's correction step (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Develop. 34(1), 1990; the division theorem of his
// "IA-64 and Elementary Functions", 2000). With r = RN(1/a) and
// q0 = RN(y r), which lies within one ulp of y / a, the remainder y - q0 a
// is a floating-point number that one FMA returns exactly, and
// RN(q0 + (y - q0 a) r) = RN(y / a). The argument holds while a, y, the
// quotient and the remainder stay in the normal range: a in [2^-20, 2^20]
// and every nonzero |y| in [2^-100, 2^100] (y = +0 gives +0 as the
// division does). The epilogue checks that per thread and tile from the
// extreme row scales and takes the IEEE division otherwise.
constexpr float kUnscaleDivisorLo = 0x1p-20f, kUnscaleDivisorHi = 0x1p20f;
// Bounds on RN(s_x s_w) that keep every nonzero y = RN(RN(float(A) s_x) s_w),
// 1 <= |A| <= 2^31, inside [2^-98, 2^98].
constexpr float kUnscaleScaleLo = 0x1p-98f, kUnscaleScaleHi = 0x1p67f;

struct Unscale {
  unsigned long long a2, nr2;  // (a, a) and (-RN(1/a), -RN(1/a))
  float a, nr;
};

__device__ __forceinline__ Unscale make_unscale(float a) {
  Unscale u;
  u.a = a;
  u.nr = -__frcp_rn(a);
  u.a2 = pair_f32(a, a);
  u.nr2 = pair_f32(u.nr, u.nr);
  return u;
}

// Whether the correction step is exact for every y of a tile whose nonzero row
// scales lie in [sx_lo, sx_hi], at weight scale sw (NaN and inf fail).
__device__ __forceinline__ bool unscale_fast_ok(float a, float sx_lo, float sx_hi, float sw) {
  const float m = fabsf(a);
  return m >= kUnscaleDivisorLo && m <= kUnscaleDivisorHi && __fmul_rn(sx_lo, sw) >= kUnscaleScaleLo &&
         __fmul_rn(sx_hi, sw) <= kUnscaleScaleHi;
}

// -RN(y / a) for both lanes of y2 (the negated form saves the negations:
// RN is symmetric, so -q0 = RN(y (-r)) and -RN(q0 + rem r) = RN(rem (-r) - q0)).
__device__ __forceinline__ unsigned long long neg_unscale_f32x2(unsigned long long y2, const Unscale& u) {
  const unsigned long long nq0 = mul_f32x2(y2, u.nr2);  // -q0
  const unsigned long long rem = f32x2_fma(nq0, u.a2, y2);  // y - q0 a, exact
  return f32x2_fma(rem, u.nr2, nq0);
}
// The IEEE division of both lanes by a, out of line: the fallback of tiles
// outside the correction step's range, kept as one call so that the unrolled
// epilogue does not carry an inlined division per element.
static __device__ __noinline__ unsigned long long unscale_div_f32x2(unsigned long long y2, float a) {
  float y0, y1;
  unpair_f32(y2, y0, y1);
  return pair_f32(__fdiv_rn(y0, a), __fdiv_rn(y1, a));
}
__device__ __forceinline__ float neg_unscale_f32(float y, const Unscale& u) {
  const float nq0 = __fmul_rn(y, u.nr);
  const float rem = __fmaf_rn(nq0, u.a, y);
  return __fmaf_rn(rem, u.nr, nq0);
}

// The smallest nonzero and the largest of 32 lanes' nonnegative fp32 values
// v[0..n) (as bit patterns, which order like the values; no nonzero value
// gives +inf as the smallest).
template <int NV>
__device__ __forceinline__ void warp_scale_range(const float (&v)[NV], float& lo, float& hi) {
  unsigned l = 0x7f800000u, h = 0u;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const unsigned b = __float_as_uint(v[k]);
    l = min(l, b ? b : 0x7f800000u);
    h = max(h, b);
  }
  lo = __uint_as_float(__reduce_min_sync(0xffffffffu, l));
  hi = __uint_as_float(__reduce_max_sync(0xffffffffu, h));
}

// End of the exact chunk that starts at K block c0 (chunks are aligned runs of
// L blocks inside a tile), clipped to kb1.
__device__ __forceinline__ int chunk_end(int c0, int L, int kb1) {
  return min(kb1, (c0 / L + 1) * L);
}

// Bounded wait until *flag == v (acquire). On giving up: sets the CTA's abort
// flag, records CONVROT_ERR_TIMEOUT and returns false.
__device__ __forceinline__ bool wait_flag(const unsigned long long* flag, unsigned long long v,
                                          volatile int* abort_flag, int* err, uint64_t limit_ns = kWaitLimitNs) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (ld_acquire_gpu(flag) == v) return true;
    if ((it & 15) == 15) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        record_error(err, CONVROT_ERR_TIMEOUT);
        return false;
      }
    }
    __nanosleep(128);
  }
}

// Raster order: tiles are taken in groups of raster_bands activation bands
// (as many as fit RASTER_L2_BYTES of codes; all of them for the usual
// shapes); inside a group, consecutive tiles walk the bands of one weight
// tile before moving to the next weight tile (of the same or the next
// linear). The group's activation codes then stay in L2 while its weight
// tiles stream through once.
__device__ __forceinline__ TileCoord decode_tile(const GemmParams& p, int t) {
  const int rb = p.raster_bands;
  const int per_group = rb * p.n_wtiles;
  const int g = t / per_group;
  const int idx = t - g * per_group;
  const int gm = min(rb, p.n_xtiles - g * rb);
  const int w = idx / gm;
  TileCoord c;
  c.xt = g * rb + (idx - w * gm);
  int j = 0;
#pragma unroll 1
  while (j + 1 < p.n_lin && w >= p.wtile_start[j + 1]) ++j;
  c.lin = j;
  c.wt = w - p.wtile_start[j];
  return c;
}

// K blocks (of BK) per exact fp32 chunk for a tile: the weight's plan for the
// tile's blocks of 128 weight rows (their minimum), or KB_PER_CHUNK (1024 products,
// always exact) without a plan.
template <int CG>
__device__ __forceinline__ int tile_chunk_kb(const GemmParams& p, const TileCoord& c) {
  int L = KB_PER_CHUNK;
  const int32_t* plan = p.kchunk[c.lin];
  if (plan) {
    const int b0 = c.wt * CG;
    const int nblk = (p.N[c.lin] + CTA_M - 1) / CTA_M;
    L = __ldg(plan + b0);
    if (CG == 2 && b0 + 1 < nblk) L = min(L, __ldg(plan + b0 + 1));
  }
  return max(1, min(L, p.num_kb));
}

// ---- host helpers (gemm.cu) ---------------------------------------------------

// fp16 [rows, K] row-major tensor map, box box_rows x 64, 128-byte swizzle.
int make_tmap(CUtensorMap* m, const void* base, int64_t rows, int64_t K, int box_rows);
// fp32 Y [rows, cols] row-major (cols % 4 == 0), box box_cols features x Y_ROWS rows.
int make_tmap_y(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_cols = CTA_M);
// Nonzero value distinct per launch for the hand-over flags.
unsigned long long next_epoch();
// Whether splitting the fractional last wave of T tiles over `units` pays.
bool split_pays(int T, int units);
// Split tiles and hand-over words for `units` co-resident units of unit_ctas CTAs.
void plan_split(GemmParams& p, int units, int unit_ctas, const GemmSync& sync);
// Launch configuration of n_units CTA pairs (clusters of two), optionally as a
// programmatic dependent of the previous kernel in the stream.
cudaLaunchConfig_t pair_config(int n_units, size_t smem, cudaStream_t stream, cudaLaunchAttribute* attr,
                               bool pdl = false);

}  // namespace gemm
}  // namespace convrot
