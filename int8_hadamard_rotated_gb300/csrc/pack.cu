// pack.cu -- the convrot activation pack on sm_103a: group-wise regular
// Hadamard rotation, per-row absmax and INT8 quantization in one pass.
//
// What it computes (stable-diffusion.cpp docs, page "INT8 Convrot
// Safetensors"): "How INT8 convrot works" gives R_G = H4^{(x)n} over every
// contiguous group of G = 4^n features; "Runtime activation quantization"
// gives s[r] = max_i |X_rot[r,i]| / 127 over the whole row and
// Q[r,i] = clamp(round(X_rot[r,i] / s[r]), -127, 127); "Weight quantization"
// applies the same rule to weight rows.
//
// Rotation. With S = diag(1,1,1,-1) and P the swap of entries 1 and 2, the
// page's H4 factors as H4 = 1/2 P S (H2 (x) H2) S, where H2 (x) H2 is the
// 4-point Walsh-Hadamard matrix. The Kronecker power therefore is
//     R_G = 2^-n  P_G S_G W_G S_G,
// with W_G the G-point Walsh-Hadamard matrix (radix-2 butterflies on the
// index bits, in any order), S_G the sign flip of every index whose count of
// base-4 digits equal to 3 is odd, and P_G the swap of the two bits of every
// base-4 digit of the index. The kernel applies the input signs, the
// butterflies, the output signs, and writes each result at its bit-swapped
// position; the 2^-n normalisation is folded exactly into the divisor.
//
// Quantizer. The code is rint(RN(z / d)) with d = s * 2^n (z / d is exactly
// X_rot / s). It is formed as q = z * RN(1/d), rounded to an integer with the
// 1.5 * 2^23 magic constant (round-half-even). |q - RN(z/d)| < 1.9e-5 for
// |z/d| <= 127.0001, so whenever q is farther than 2^-15 from a half-integer
// both round to the same integer; the rare values nearer than that are
// recomputed with the IEEE division. |z/d| <= 127 (1 + 2^-23) because d is
// max|z| / 127 rounded once, so the rounded code already lies in [-127, 127]
// and the clamp of the definition never changes it.
//
// Data layout. A thread owns 64 elements of one row: four "units" of 16
// consecutive elements (index bits 0-3 in registers). For G >= 64 the four
// units are the four values of the group's top base-4 digit (registers); the
// digits between bit 4 and the top digit live on G/64 consecutive lanes
// (shuffles). A row is handled by ceil(K/64) threads of one CTA.
//
// Pipeline. CTAs are persistent over blocks of rows. Each thread prefetches
// its next block with 16-byte cp.async copies into a private, lane-interleaved
// shared-memory layout ([stage][chunk][thread], conflict-free), so one block's
// loads are in flight while the previous one is rotated and quantized. The row
// absmax is a warp-segment shuffle reduction plus one shared-memory 64-bit
// atomic max per segment, tagged with the iteration so no reset is needed.
#include "common.cuh"

#include <algorithm>
#include <mutex>

namespace convrot {
namespace {

template <int G>
struct Geo {
  static constexpr int kLog2G = (G == 1) ? 0 : (G == 4) ? 2 : (G == 16) ? 4 : (G == 64) ? 6 : (G == 256) ? 8 : 10;
  static constexpr int kTPG = (G >= 64) ? G / 64 : 1;                 // threads per group
  static constexpr int kLaneBits = (G == 256) ? 2 : (G == 1024) ? 4 : 0;
  static constexpr int kUnitBits = (kLog2G < 4) ? kLog2G : 4;          // butterfly bits inside a unit
  static constexpr bool kUnitDigit = (G >= 64);                        // the 4 units form one digit
  static constexpr float kInvScale = 1.0f / float(1 << (kLog2G / 2));  // 2^-n
  static constexpr float kScale = float(1 << (kLog2G / 2));            // 2^n
};

__host__ __device__ constexpr int swap2(int x) { return ((x & 1) << 1) | ((x >> 1) & 1); }
__host__ __device__ constexpr int swap_digit_bits4(int x) { return swap2(x & 3) | (swap2((x >> 2) & 3) << 2); }

// Static part of the sign S_G at in-register coordinates (unit j, position p):
// 1 when the number of base-4 digits equal to 3 among the register digits is odd.
template <int G>
__host__ __device__ constexpr int static_sign(int j, int p) {
  int c = 0;
  if (G >= 4) c += ((p & 3) == 3);
  if (G >= 16) c += (((p >> 2) & 3) == 3);
  if (G >= 64) c += (j == 3);
  return c & 1;
}
// Lane part of S_G for lane-in-group li.
template <int G>
__host__ __device__ constexpr int lane_sign(int li) {
  int c = 0;
  if (G >= 256) c += ((li & 3) == 3);
  if (G >= 1024) c += (((li >> 2) & 3) == 3);
  return c & 1;
}

// Output position (inside its unit) of the value held at position p.
template <int G>
__host__ __device__ constexpr int out_pos(int p) {
  return (G == 1) ? p : (G == 4) ? ((p & ~3) | swap2(p & 3)) : swap_digit_bits4(p);
}

// ---- packed fp32x2 arithmetic (sm_100+) -------------------------------------
__device__ __forceinline__ unsigned long long f2pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2unpack(unsigned long long r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long sub2(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// Radix-2 butterfly on two packed pairs: (a, b) -> (a + b, a - b), lane-wise.
__device__ __forceinline__ void bfly2(unsigned long long& a, unsigned long long& b) {
  const unsigned long long s = add2(a, b);
  b = sub2(a, b);
  a = s;
}

// ---- cp.async ----------------------------------------------------------------
__device__ __forceinline__ void cp_async16(uint32_t dst_smem, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst_smem), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack4_low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  const uint32_t lo = __byte_perm(a, b, 0x0040);
  const uint32_t hi = __byte_perm(c, d, 0x0040);
  return __byte_perm(lo, hi, 0x5410);
}

constexpr int kMaxThreads = 512;
constexpr int kMaxRowsPerCta = 256;
constexpr float kMagic = 12582912.0f;        // 1.5 * 2^23
constexpr float kNearHalf = 0.5f - 1.0f / 32768.0f;  // 0.5 - 2^-15

template <typename TIn>
struct InTraits;
template <>
struct InTraits<float> {
  static constexpr int kChunksPerUnit = 4;  // 16 fp32 = 64 B = 4 x 16 B
};
template <>
struct InTraits<__half> {
  static constexpr int kChunksPerUnit = 2;  // 16 fp16 = 32 B = 2 x 16 B
};

// Convert the 16-byte chunks of one unit (as loaded) to 16 fp32 values.
template <typename TIn>
__device__ __forceinline__ void unit_to_f32(const uint4 (&c)[InTraits<TIn>::kChunksPerUnit], float (&v)[16]);

template <>
__device__ __forceinline__ void unit_to_f32<float>(const uint4 (&c)[4], float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[4 * i + 0] = __uint_as_float(c[i].x);
    v[4 * i + 1] = __uint_as_float(c[i].y);
    v[4 * i + 2] = __uint_as_float(c[i].z);
    v[4 * i + 3] = __uint_as_float(c[i].w);
  }
}
template <>
__device__ __forceinline__ void unit_to_f32<__half>(const uint4 (&c)[2], float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t w[4] = {c[i].x, c[i].y, c[i].z, c[i].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __half2 h = *reinterpret_cast<const __half2*>(&w[k]);
      float2 f = __half22float2(h);
      v[8 * i + 2 * k] = f.x;
      v[8 * i + 2 * k + 1] = f.y;
    }
  }
}

// One CTA handles `rpc` rows with `tpr` threads each per block, persistently.
template <int G, typename TIn, int OUT>
__global__ void __launch_bounds__(kMaxThreads)
pack_kernel(const TIn* __restrict__ X, int64_t M, int K, int tpr, int rpc, int64_t nblocks,
            int two_stage, void* __restrict__ out_codes, float* __restrict__ scales) {
  using C = Geo<G>;
  constexpr int CPU = InTraits<TIn>::kChunksPerUnit;
  constexpr int CH = 4 * CPU;  // 16-byte chunks per thread per stage
  extern __shared__ uint4 stage_buf[];  // [1 or 2][CH][blockDim.x]
  __shared__ unsigned long long s_amax[2][kMaxRowsPerCta];

  const int tid = threadIdx.x;
  const int nth = blockDim.x;
  const int lr = tid / tpr;
  const int t = tid - lr * tpr;
  const int units = K >> 4;
  const int gi = t / C::kTPG;
  const int li = t - gi * C::kTPG;
  const bool in_cta_row = lr < rpc;

  for (int i = tid; i < 2 * kMaxRowsPerCta; i += nth) (&s_amax[0][0])[i] = 0ull;

  const uint32_t sbase = smem_u32(stage_buf);
  auto issue = [&](int64_t blk, int stage) {
    const int64_t row = blk * rpc + lr;
    const bool active = in_cta_row && row < M;
    const TIn* xrow = X + (active ? row : 0) * static_cast<int64_t>(K);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int u = gi * 4 * C::kTPG + j * C::kTPG + li;
      const bool ok = active && u < units;
      const TIn* src = ok ? xrow + 16 * u : X;
#pragma unroll
      for (int c = 0; c < CPU; ++c) {
        const uint32_t dst = sbase + static_cast<uint32_t>(((stage * CH + j * CPU + c) * nth + tid) * 16);
        cp_async16(dst, ok ? static_cast<const void*>(reinterpret_cast<const uint4*>(src) + c)
                           : static_cast<const void*>(src),
                   ok ? 16u : 0u);
      }
    }
  };

  // lane-sign bookkeeping for the cross-lane butterflies (see below)
  float lane_coef[C::kLaneBits > 0 ? C::kLaneBits : 1];
  int rho_mask = 0;
#pragma unroll
  for (int b = 0; b < C::kLaneBits; ++b) {
    const int pli = li ^ (1 << b);
    const int rs = lane_sign<G>(li ^ rho_mask);
    const int rp = lane_sign<G>(pli ^ rho_mask);
    const int sb = (li >> b) & 1;
    lane_coef[b] = ((sb ^ rs ^ rp) & 1) ? -1.0f : 1.0f;
    rho_mask |= (1 << b);
  }
  // residual lane sign of the held values, times the output lane sign
  const int lane_flip = (C::kLaneBits > 0) ? (lane_sign<G>(li ^ rho_mask) ^ lane_sign<G>(li)) : 0;

  // aligned lane segments of gcd(tpr, 32) lanes never straddle two rows
  const int seg = tpr & -tpr;
  const int segw = seg < 32 ? seg : 32;

  __syncthreads();  // s_amax initialised

  int64_t blk = blockIdx.x;
  if (blk < nblocks) issue(blk, 0);
  cp_async_commit();
  for (uint32_t it = 0; blk < nblocks; blk += gridDim.x, ++it) {
    const int stage = two_stage ? static_cast<int>(it & 1) : 0;
    if (two_stage) {
      if (blk + gridDim.x < nblocks) issue(blk + gridDim.x, stage ^ 1);
      cp_async_commit();
      cp_async_wait_1();
    } else {
      if (it > 0) {
        issue(blk, 0);
        cp_async_commit();
      }
      cp_async_wait_0();
    }

    const int64_t row = blk * rpc + lr;
    const bool active = in_cta_row && row < M;

    // ---- load own data from shared memory --------------------------------
    float v[4][16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint4 c[CPU];
#pragma unroll
      for (int k = 0; k < CPU; ++k) c[k] = stage_buf[(stage * CH + j * CPU + k) * nth + tid];
      unit_to_f32<TIn>(c, v[j]);
    }

    // ---- input signs of the register digits ------------------------------
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int p = 0; p < 16; ++p)
        if (static_sign<G>(j, p)) v[j][p] = -v[j][p];

    // ---- butterflies: bit 0 scalar, then packed pairs (p, p+1) ------------
    if (C::kUnitBits >= 1) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int p = 0; p < 16; p += 2) {
          const float a = v[j][p], c = v[j][p + 1];
          v[j][p] = a + c;
          v[j][p + 1] = a - c;
        }
    }
    unsigned long long w[4][8];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int h = 0; h < 8; ++h) w[j][h] = f2pack(v[j][2 * h], v[j][2 * h + 1]);
#pragma unroll
    for (int b = 1; b < C::kUnitBits; ++b) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int h = 0; h < 8; ++h)
          if (!((h >> (b - 1)) & 1)) bfly2(w[j][h], w[j][h | (1 << (b - 1))]);
    }
    if (C::kUnitDigit) {
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (!((j >> b) & 1))
#pragma unroll
            for (int h = 0; h < 8; ++h) bfly2(w[j][h], w[j | (1 << b)][h]);
    }
    // ---- butterflies across lanes ----------------------------------------
    // The true value is rho * held. A butterfly on lane bit b maps
    //   true' = (bit ? -1 : 1) * true(self) + true(partner)
    // to held' = fma(held, s_b * rho(self) * rho(partner), held(partner)) and
    // rho'(self) = rho(partner); the coefficients are per-lane constants.
#pragma unroll
    for (int b = 0; b < C::kLaneBits; ++b) {
      const unsigned long long cc = f2pack(lane_coef[b], lane_coef[b]);
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          float a0, a1;
          f2unpack(w[j][h], a0, a1);
          const float u0 = __shfl_xor_sync(0xffffffffu, a0, 1 << b);
          const float u1 = __shfl_xor_sync(0xffffffffu, a1, 1 << b);
          w[j][h] = fma2(w[j][h], cc, f2pack(u0, u1));
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int h = 0; h < 8; ++h) f2unpack(w[j][h], v[j][2 * h], v[j][2 * h + 1]);

    // ---- row absmax ----------------------------------------------------------
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int p = 0; p < 16; ++p) amax = fmaxf(amax, fabsf(v[j][p]));
    unsigned abits = __float_as_uint(amax);
#pragma unroll
    for (int off = 1; off < 32; off <<= 1)
      if (off < segw) abits = max(abits, __shfl_xor_sync(0xffffffffu, abits, off));
    const unsigned long long tag = static_cast<unsigned long long>(it + 1) << 32;
    const int slot = it & 1;
    if (active && (t % segw) == 0) atomicMax(&s_amax[slot][lr], tag | abits);
    __syncthreads();
    if (!active) continue;

    const float amax_z = __uint_as_float(static_cast<unsigned>(s_amax[slot][lr] & 0xffffffffull));
    // X_rot = z * 2^-n exactly, so max |X_rot| = amax_z * 2^-n.
    const float s = __fdiv_rn(amax_z * C::kInvScale, 127.0f);
    if (t == 0) scales[row] = s;
    // z / (s * 2^n) equals X_rot / s as a real number, hence the same rounded quotient.
    float d = s * C::kScale;
    if (lane_flip) d = -d;
    const bool zero_row = (s == 0.0f);
    const float rcp = zero_row ? 0.0f : __frcp_rn(d);
    const unsigned long long rcp2 = f2pack(rcp, rcp);
    const unsigned long long magic2 = f2pack(kMagic, kMagic);

    // ---- quantize and store ----------------------------------------------------
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int u = gi * 4 * C::kTPG + j * C::kTPG + li;
      if (u >= units) continue;
      int uo;
      if (G <= 16) uo = u;
      else if (G == 64) uo = gi * 4 + swap2(j);
      else if (G == 256) uo = gi * 16 + swap2(j) * 4 + swap2(li);
      else uo = gi * 64 + swap2(j) * 16 + swap_digit_bits4(li);
      float qr[16];   // rounded codes as floats (integers), in output order
      bool near_half = false;
#pragma unroll
      for (int p = 0; p < 16; p += 2) {
        // output sign of the register digits (same function as the input sign)
        const float z0 = static_sign<G>(j, p) ? -v[j][p] : v[j][p];
        const float z1 = static_sign<G>(j, p + 1) ? -v[j][p + 1] : v[j][p + 1];
        const unsigned long long q = mul2(f2pack(z0, z1), rcp2);
        const unsigned long long t2 = sub2(add2(q, magic2), magic2);
        const unsigned long long e = sub2(q, t2);
        float e0, e1, t0, t1;
        f2unpack(e, e0, e1);
        f2unpack(t2, t0, t1);
        near_half |= (fabsf(e0) > kNearHalf) | (fabsf(e1) > kNearHalf);
        qr[out_pos<G>(p)] = t0;
        qr[out_pos<G>(p + 1)] = t1;
      }
      if (near_half) {
        // exact IEEE quotient for the values near a rounding boundary
#pragma unroll
        for (int p = 0; p < 16; ++p) {
          const float z = static_sign<G>(j, p) ? -v[j][p] : v[j][p];
          const float q = z * rcp;
          const float tt = (q + kMagic) - kMagic;
          if (fabsf(q - tt) > kNearHalf) qr[out_pos<G>(p)] = rintf(__fdiv_rn(z, d));
        }
      }
      if (zero_row) {
#pragma unroll
        for (int p = 0; p < 16; ++p) qr[p] = 0.0f;
      }
      if (OUT == kPackI8) {
        int8_t* dst = static_cast<int8_t*>(out_codes) + row * static_cast<int64_t>(K) + 16 * uo;
        uint32_t b[16];
#pragma unroll
        for (int p = 0; p < 16; ++p) b[p] = __float_as_uint(qr[p] + kMagic);  // low byte = code
        uint4 wv;
        wv.x = pack4_low_bytes(b[0], b[1], b[2], b[3]);
        wv.y = pack4_low_bytes(b[4], b[5], b[6], b[7]);
        wv.z = pack4_low_bytes(b[8], b[9], b[10], b[11]);
        wv.w = pack4_low_bytes(b[12], b[13], b[14], b[15]);
        *reinterpret_cast<uint4*>(dst) = wv;
      } else {
        __half* dst = static_cast<__half*>(out_codes) + row * static_cast<int64_t>(K) + 16 * uo;
        uint32_t hw[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          __half2 h = __floats2half2_rn(qr[2 * k], qr[2 * k + 1]);
          hw[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        reinterpret_cast<uint4*>(dst)[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        reinterpret_cast<uint4*>(dst)[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
      }
    }
  }
}

int gcd_int(int a, int b) { while (b) { int t = a % b; a = b; b = t; } return a; }

template <int G, typename TIn, int OUT>
int launch_pack_t(const void* X, int64_t M, int K, void* out, float* scales, cudaStream_t stream) {
  const int tpr = (K + 63) / 64;
  int rpc = 32 / gcd_int(tpr, 32);
  int threads = tpr * rpc;
  if (threads > kMaxThreads) {
    rpc = 1;
    threads = ((tpr + 31) / 32) * 32;
  }
  while (threads * 2 <= 256 && tpr * rpc * 2 <= kMaxThreads && rpc * 2 <= kMaxRowsPerCta) {
    rpc *= 2;
    threads = ((tpr * rpc + 31) / 32) * 32;
  }
  constexpr int CH = 4 * InTraits<TIn>::kChunksPerUnit;
  constexpr size_t kSmemLimit = 200 * 1024;  // leaves room for the static shared memory
  const int two_stage = (static_cast<size_t>(2) * CH * threads * 16 <= kSmemLimit) ? 1 : 0;
  const size_t smem = static_cast<size_t>(two_stage ? 2 : 1) * CH * threads * 16;
  auto kern = pack_kernel<G, TIn, OUT>;
  static std::mutex mu;
  static size_t configured_smem = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (smem > configured_smem) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return set_cuda_error(e);
      configured_smem = smem;
    }
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
  if (e != cudaSuccess) return set_cuda_error(e);
  if (per_sm < 1) per_sm = 1;
  const int64_t nblocks = (M + rpc - 1) / rpc;
  const int64_t grid = std::min<int64_t>(nblocks, static_cast<int64_t>(per_sm) * device_sm_count());
  pack_kernel<G, TIn, OUT><<<static_cast<unsigned>(grid), threads, smem, stream>>>(
      static_cast<const TIn*>(X), M, K, tpr, rpc, nblocks, two_stage, out, scales);
  return check_launch();
}

template <typename TIn, int OUT>
int dispatch_group(const void* X, int64_t M, int K, int G, void* out, float* scales, cudaStream_t s) {
  switch (G) {
    case 1: return launch_pack_t<1, TIn, OUT>(X, M, K, out, scales, s);
    case 4: return launch_pack_t<4, TIn, OUT>(X, M, K, out, scales, s);
    case 16: return launch_pack_t<16, TIn, OUT>(X, M, K, out, scales, s);
    case 64: return launch_pack_t<64, TIn, OUT>(X, M, K, out, scales, s);
    case 256: return launch_pack_t<256, TIn, OUT>(X, M, K, out, scales, s);
    case 1024: return launch_pack_t<1024, TIn, OUT>(X, M, K, out, scales, s);
    default: return CONVROT_ERR_GROUP;
  }
}

__device__ __forceinline__ uint32_t pack2_f16(int q0, int q1) {
  __half2 h = __halves2half2(__int2half_rn(q0), __int2half_rn(q1));
  return *reinterpret_cast<uint32_t*>(&h);
}

// int8 -> fp16 codes, 16 elements per thread.
__global__ void __launch_bounds__(256) widen_kernel(const int8_t* __restrict__ src,
                                                    __half* __restrict__ dst, int64_t n16) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n16) return;
  const uint4 a = __ldcs(reinterpret_cast<const uint4*>(src) + i);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
  uint32_t h[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int b0 = static_cast<int8_t>(w[k] & 0xff), b1 = static_cast<int8_t>((w[k] >> 8) & 0xff);
    const int b2 = static_cast<int8_t>((w[k] >> 16) & 0xff), b3 = static_cast<int8_t>(w[k] >> 24);
    h[2 * k] = pack2_f16(b0, b1);
    h[2 * k + 1] = pack2_f16(b2, b3);
  }
  uint4* d = reinterpret_cast<uint4*>(dst) + 2 * i;
  d[0] = make_uint4(h[0], h[1], h[2], h[3]);
  d[1] = make_uint4(h[4], h[5], h[6], h[7]);
}

}  // namespace

int launch_pack(const void* X, int x_dtype, int64_t M, int64_t K, int G,
                void* out_codes, int out_kind, float* scales, cudaStream_t stream) {
  if (M == 0) return CONVROT_OK;
  const int k = static_cast<int>(K);
  if (x_dtype == CONVROT_F32) {
    return out_kind == kPackI8 ? dispatch_group<float, kPackI8>(X, M, k, G, out_codes, scales, stream)
                               : dispatch_group<float, kPackF16>(X, M, k, G, out_codes, scales, stream);
  }
  return out_kind == kPackI8 ? dispatch_group<__half, kPackI8>(X, M, k, G, out_codes, scales, stream)
                             : dispatch_group<__half, kPackF16>(X, M, k, G, out_codes, scales, stream);
}

int launch_widen(const int8_t* src, __half* dst, int64_t n, cudaStream_t stream) {
  if (n == 0) return CONVROT_OK;
  const int64_t n16 = n / 16;
  const int64_t blocks = (n16 + 255) / 256;
  widen_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(src, dst, n16);
  return check_launch();
}

}  // namespace convrot
