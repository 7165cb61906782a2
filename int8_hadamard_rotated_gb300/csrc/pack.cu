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
// recomputed as rint(RN(RN(z 2^-n) / s)), the definition's two roundings
// (RN(z 2^-n) is X_rot itself, exact unless X_rot is subnormal). When s is a
// normal float, |z/d| <= 127 (1 + 2^-23) because d is max|z| / 127 rounded
// once, so the rounded code already lies in [-127, 127] and the clamp of the
// definition never changes it. A row whose s is subnormal (max |X_rot| below
// about 127 * 2^-126) has lost precision in s, so codes beyond 127 can occur
// and 1/d can overflow: every code of such a row takes the definition's
// division and clamp.
//
// Data layout. A thread owns 64 elements of one row: four "units" of 16
// consecutive elements (index bits 0-3 in registers). For G >= 64 the four
// units are the four values of the group's top base-4 digit (registers); the
// digits between bit 4 and the top digit live on G/64 consecutive lanes
// (shuffles). For G <= 16 every unit is a whole number of groups, so units
// are dealt out to the row's threads round-robin. A row is handled by
// ceil(K/64) threads of one CTA; the row absmax is a warp-segment shuffle
// reduction plus one shared-memory 64-bit atomic max per segment, tagged with
// the iteration so no reset is needed.
//
// Two kernels share that arithmetic:
//   pack_tma_kernel (rows whose length is a whole number of 128-byte lines):
//     persistent CTAs over blocks of R rows. One thread streams blocks into a
//     ring of shared-memory stages with 3-D TMA tensor copies (128-byte
//     swizzle, so the threads' 16-byte reads of their units spread over the
//     banks); the codes of a block are staged in shared memory and written
//     back with one bulk copy, while the next blocks' loads are in flight.
//   pack_kernel (any K % 16 == 0, rows up to 32768 elements): per-thread
//     16-byte cp.async copies into a lane-interleaved two-stage buffer and
//     direct 16-byte stores of the codes.
// A prologue may transform each loaded row first: GELU, or the modulation
// (RMS norm, per-channel weight, (x + x*scale) + shift). The modulated pack takes
// pack_tma_kernel for rows of up to kVecSmemMaxK features, with the three
// modulation vectors staged once per CTA in shared memory, and pack_kernel
// for longer rows.
#include "common.cuh"

#include <algorithm>
#include <cstring>
#include <mutex>

namespace convrot {

// Sticky device error word of the pack kernels (timeouts of bounded waits).
__device__ int g_pack_error = 0;

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
constexpr float kMinNormal = 1.17549435082228751e-38f;  // 2^-126, the smallest normal float

// Parameters of the modulation prologue (kProModulate).
struct ModPrologue {
  const float* weight;  // [K] per-channel multiplier after the norm, or null
  const float* scale;   // [K] modulation scale: (x + x * scale), or null
  const float* shift;   // [K] modulation shift: + shift, or null
  float eps;            // RMS norm epsilon
  int rms;              // 1: divide each row by sqrt(mean(x^2) + eps) first
};

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


// ---- the per-thread arithmetic shared by both kernels ------------------------

// Per-lane constants of the cross-lane butterflies (G = 256, 1024). The true
// value of a held number is rho * held. A butterfly on lane bit b maps
//   true' = (bit ? -1 : 1) * true(self) + true(partner)
// to held' = fma(held, coef[b], held(partner)) with
// coef[b] = s_b * rho(self) * rho(partner), and rho'(self) = rho(partner);
// the coefficients are per-lane constants. `flip` is the residual rho of the
// held values times the lane's output sign.
template <int G>
struct LaneSigns {
  float coef[Geo<G>::kLaneBits > 0 ? Geo<G>::kLaneBits : 1];
  int flip;
};

template <int G>
__device__ __forceinline__ LaneSigns<G> lane_signs(int li) {
  LaneSigns<G> ls;
  int rho_mask = 0;
#pragma unroll
  for (int b = 0; b < Geo<G>::kLaneBits; ++b) {
    const int pli = li ^ (1 << b);
    const int rs = lane_sign<G>(li ^ rho_mask);
    const int rp = lane_sign<G>(pli ^ rho_mask);
    const int sb = (li >> b) & 1;
    ls.coef[b] = ((sb ^ rs ^ rp) & 1) ? -1.0f : 1.0f;
    rho_mask |= (1 << b);
  }
  if (Geo<G>::kLaneBits == 0) ls.coef[0] = 1.0f;
  ls.flip = (Geo<G>::kLaneBits > 0) ? (lane_sign<G>(li ^ rho_mask) ^ lane_sign<G>(li)) : 0;
  return ls;
}

// Input signs and every butterfly of W_G on the 64 values a thread holds
// (in place). The result is 2^n X_rot up to the lane sign `flip`, with the
// output signs of the register digits still to be applied.
template <int G>
__device__ __forceinline__ void rotate64(float (&v)[4][16], const LaneSigns<G>& ls) {
  using C = Geo<G>;
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int p = 0; p < 16; ++p)
      if (static_sign<G>(j, p)) v[j][p] = -v[j][p];

  // bit 0 scalar, then packed pairs (p, p+1)
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
#pragma unroll
  for (int b = 0; b < C::kLaneBits; ++b) {
    const unsigned long long cc = f2pack(ls.coef[b], ls.coef[b]);
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
}

__device__ __forceinline__ float absmax64(const float (&v)[4][16]) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int p = 0; p < 16; ++p) amax = fmaxf(amax, fabsf(v[j][p]));
  return amax;
}

// Divisor of the held values: d = s * 2^n (negated when the lane's held values
// carry a residual sign), so that z / d = X_rot / s as real numbers.
template <int G>
__device__ __forceinline__ float held_divisor(float s, int flip) {
  const float d = s * Geo<G>::kScale;
  return flip ? -d : d;
}

// The code of held value z by the definition: rint(X_rot / s) with
// X_rot = RN(z 2^-n) and s = d 2^-n (exact: a power-of-two scaling of the
// divisor, sign included), clamped to [-127, 127].
template <int G>
__device__ __forceinline__ float exact_code(float z, float d) {
  const float q = rintf(__fdiv_rn(__fmul_rn(z, Geo<G>::kInvScale), __fmul_rn(d, Geo<G>::kInvScale)));
  return fminf(fmaxf(q, -127.0f), 127.0f);
}

// Codes of unit j (rounded quotients as integer-valued floats), in output order.
// tiny_row: s is subnormal, so every code takes the definition's division.
template <int G>
__device__ __forceinline__ void quantize_unit(const float (&vj)[16], int j, float d, float rcp, bool zero_row,
                                              bool tiny_row, float (&qr)[16]) {
  if (tiny_row) {
#pragma unroll
    for (int p = 0; p < 16; ++p) qr[out_pos<G>(p)] = exact_code<G>(static_sign<G>(j, p) ? -vj[p] : vj[p], d);
    return;
  }
  const unsigned long long rcp2 = f2pack(rcp, rcp);
  const unsigned long long magic2 = f2pack(kMagic, kMagic);
  bool near_half = false;
#pragma unroll
  for (int p = 0; p < 16; p += 2) {
    // output sign of the register digits (the same function as the input sign)
    const float z0 = static_sign<G>(j, p) ? -vj[p] : vj[p];
    const float z1 = static_sign<G>(j, p + 1) ? -vj[p + 1] : vj[p + 1];
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
    // the exact IEEE quotient for the values near a rounding boundary
#pragma unroll
    for (int p = 0; p < 16; ++p) {
      const float z = static_sign<G>(j, p) ? -vj[p] : vj[p];
      const float q = z * rcp;
      const float tt = (q + kMagic) - kMagic;
      if (fabsf(q - tt) > kNearHalf) qr[out_pos<G>(p)] = exact_code<G>(z, d);
    }
  }
  if (zero_row) {
#pragma unroll
    for (int p = 0; p < 16; ++p) qr[p] = 0.0f;
  }
}

// 16 codes -> 16 int8 bytes (one 16-byte vector).
__device__ __forceinline__ uint4 codes_i8(const float (&qr)[16]) {
  uint32_t b[16];
#pragma unroll
  for (int p = 0; p < 16; ++p) b[p] = __float_as_uint(qr[p] + kMagic);  // low byte = code
  uint4 wv;
  wv.x = pack4_low_bytes(b[0], b[1], b[2], b[3]);
  wv.y = pack4_low_bytes(b[4], b[5], b[6], b[7]);
  wv.z = pack4_low_bytes(b[8], b[9], b[10], b[11]);
  wv.w = pack4_low_bytes(b[12], b[13], b[14], b[15]);
  return wv;
}

// 16 codes -> 16 binary16 integers (two 16-byte vectors).
__device__ __forceinline__ void codes_f16(const float (&qr)[16], uint4& lo, uint4& hi) {
  uint32_t hw[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    __half2 h = __floats2half2_rn(qr[2 * k], qr[2 * k + 1]);
    hw[k] = *reinterpret_cast<uint32_t*>(&h);
  }
  lo = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  hi = make_uint4(hw[4], hw[5], hw[6], hw[7]);
}

// Unit of the row held in register slot j by a thread (gi, li); and the unit
// its codes are written to (the bit-swap permutation P_G acts on the digits
// above bit 3 here, and on bits 0-3 through out_pos).
template <int G>
__device__ __forceinline__ int in_unit_grouped(int gi, int li, int j) {
  return gi * 4 * Geo<G>::kTPG + j * Geo<G>::kTPG + li;
}
template <int G>
__device__ __forceinline__ int out_unit(int u, int gi, int li, int j) {
  if (G <= 16) return u;
  if (G == 64) return gi * 4 + swap2(j);
  if (G == 256) return gi * 16 + swap2(j) * 4 + swap2(li);
  return gi * 64 + swap2(j) * 16 + swap_digit_bits4(li);
}

// An input scale other than 1: every element is multiplied by it (one fp32
// rounding) before the rotation.
__device__ __forceinline__ void scale_unit(float (&v)[16], float a) {
#pragma unroll
  for (int p = 0; p < 16; ++p) v[p] = __fmul_rn(v[p], a);
}

// Prologue applied to the loaded rows before the rotation: none, GELU (the
// MLP's activation, gelu_as2, applied where its output is quantized for the
// down linear), or the modulation (per-row RMS norm, per-channel weight,
// (x + x*scale) + shift).
constexpr int kProNone = 0;
constexpr int kProGelu = 1;
constexpr int kProModulate = 2;  // per-row RMS norm and per-channel weight / modulation (ModPrologue)

template <int PRO>
__device__ __forceinline__ void prologue_unit(float (&v)[16]) {
  if (PRO == kProGelu) {
#pragma unroll
    for (int p = 0; p < 16; p += 2) gelu_as2(v[p], v[p + 1]);
  }
}

// A row's sum of squares from the partial sums of its lane segments, stored
// at part[0 .. nseg-1] by the segment leaders, added in segment order (so the
// result does not depend on which segment finished first).
__device__ __forceinline__ float row_sumsq(const float* part, int nseg) {
  float tot = 0.0f;
  for (int q = 0; q < nseg; ++q) tot += part[q];
  return tot;
}

// 1 / sqrt(sum / K + eps) of a row from its sum of squares (IEEE fp32 steps).
__device__ __forceinline__ float rms_factor(float sumsq, int K, float eps) {
  const float mean = __fdiv_rn(sumsq, static_cast<float>(K));
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
}

// The modulation vectors staged in shared memory: the 48 16-byte chunks a
// thread at position t of its row uses (chunk c of unit slot j of vector k:
// 0 weight, 1 scale, 2 shift) are consecutive from t * kModStride. The one
// chunk of padding makes lanes t .. t+7 start 196 words apart, on distinct
// banks, and every read is a per-thread base plus a constant offset.
constexpr int kModStride = 49;
__device__ __forceinline__ int mod_slot(int k, int j, int c) { return (k * 4 + j) * 4 + c; }

// Chunk c (features 4c .. 4c+3 of unit u) of modulation vector k, from global memory.
__device__ __forceinline__ float4 mod_chunk_global(const ModPrologue& m, int k, int u, int c) {
  const float* base = (k == 0) ? m.weight : (k == 1) ? m.scale : m.shift;
  return __ldg(reinterpret_cast<const float4*>(base + 16 * u) + c);
}

// The per-channel part of the modulation prologue on one unit: x * r, then
// * weight, then (x + x * scale) + shift, each operation one fp32 rounding
// (lane-wise pairs, each lane rounded as the scalar operation); absent parts
// are skipped. chunk(k, c) gives the unit's chunk c of vector k.
template <typename Chunk>
__device__ __forceinline__ void modulate_unit(float (&v)[16], float r, bool rms, const ModPrologue& m, Chunk chunk) {
  const unsigned long long r2 = f2pack(r, r);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    unsigned long long lo = f2pack(v[4 * c], v[4 * c + 1]);
    unsigned long long hi = f2pack(v[4 * c + 2], v[4 * c + 3]);
    if (rms) {
      lo = mul2(lo, r2);
      hi = mul2(hi, r2);
    }
    if (m.weight) {
      const float4 w = chunk(0, c);
      lo = mul2(lo, f2pack(w.x, w.y));
      hi = mul2(hi, f2pack(w.z, w.w));
    }
    if (m.scale) {
      const float4 q = chunk(1, c);
      lo = add2(lo, mul2(lo, f2pack(q.x, q.y)));
      hi = add2(hi, mul2(hi, f2pack(q.z, q.w)));
    }
    if (m.shift) {
      const float4 h = chunk(2, c);
      lo = add2(lo, f2pack(h.x, h.y));
      hi = add2(hi, f2pack(h.z, h.w));
    }
    f2unpack(lo, v[4 * c], v[4 * c + 1]);
    f2unpack(hi, v[4 * c + 2], v[4 * c + 3]);
  }
}

// Sum of squares of the 64 values a thread holds, reduced over the lanes of
// its row segment.
__device__ __forceinline__ float row_sumsq_part(const float (&v)[4][16], int segw) {
  // four independent lane-wise pair sums (short dependency chains), then their total
  unsigned long long acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int p = 0; p < 16; p += 2) {
      const unsigned long long x = f2pack(v[j][p], v[j][p + 1]);
      acc[j] = fma2(x, x, acc[j]);
    }
  const unsigned long long a2 = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
  float s0, s1;
  f2unpack(a2, s0, s1);
  float ss = s0 + s1;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1)
    if (off < segw) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  return ss;
}

// Lane segments per row: a row's tpr threads form aligned segments of
// gcd(tpr, 32) lanes.
__host__ __device__ constexpr int row_segments(int tpr) { return tpr / ((tpr & -tpr) < 32 ? (tpr & -tpr) : 32); }

// ---- pack_kernel: the general path (per-thread cp.async) ---------------------

// One CTA handles `rpc` rows with `tpr` threads each per block, persistently.
template <int G, typename TIn, int OUT, int PRO>
__global__ void __launch_bounds__(kMaxThreads)
pack_kernel(const TIn* __restrict__ X, int64_t M, int K, int tpr, int rpc, int64_t nblocks,
            int two_stage, float in_scale, ModPrologue mod, void* __restrict__ out_codes,
            float* __restrict__ scales) {
  using C = Geo<G>;
  constexpr int CPU = InTraits<TIn>::kChunksPerUnit;
  constexpr int CH = 4 * CPU;  // 16-byte chunks per thread per stage
  extern __shared__ uint4 stage_buf[];  // [1 or 2][CH][blockDim.x]
  __shared__ unsigned long long s_amax[2][kMaxRowsPerCta];
  __shared__ float s_sumsq[kMaxThreads];  // [rpc][segments per row]: partial sums of squares

  const int tid = threadIdx.x;
  const int nth = blockDim.x;
  const int lr = tid / tpr;
  const int t = tid - lr * tpr;
  const int units = K >> 4;
  const int gi = t / C::kTPG;
  const int li = t - gi * C::kTPG;
  const bool in_cta_row = lr < rpc;

  pdl_launch_dependents();  // the next kernel may set itself up; it waits for this one before reading
  for (int i = tid; i < 2 * kMaxRowsPerCta; i += nth) (&s_amax[0][0])[i] = 0ull;

  const uint32_t sbase = smem_u32(stage_buf);
  auto issue = [&](int64_t blk, int stage) {
    const int64_t row = blk * rpc + lr;
    const bool active = in_cta_row && row < M;
    const TIn* xrow = X + (active ? row : 0) * static_cast<int64_t>(K);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int u = in_unit_grouped<G>(gi, li, j);
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

  const LaneSigns<G> ls = lane_signs<G>(li);
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

    float v[4][16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint4 c[CPU];
#pragma unroll
      for (int k = 0; k < CPU; ++k) c[k] = stage_buf[(stage * CH + j * CPU + k) * nth + tid];
      unit_to_f32<TIn>(c, v[j]);
      prologue_unit<PRO>(v[j]);
      if (in_scale != 1.0f) scale_unit(v[j], in_scale);
    }
    const int slot = it & 1;
    if (PRO == kProModulate) {
      float r = 1.0f;
      if (mod.rms) {
        // one slot per lane segment (the previous block's reads ended before
        // the barrier that follows its row maximum)
        const int nseg = tpr / segw;
        const float ss = row_sumsq_part(v, segw);
        if (active && (t % segw) == 0) s_sumsq[lr * nseg + t / segw] = ss;
        __syncthreads();
        r = rms_factor(row_sumsq(s_sumsq + (in_cta_row ? lr : 0) * nseg, nseg), K, mod.eps);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int u = in_unit_grouped<G>(gi, li, j);
        if (active && u < units)
          modulate_unit(v[j], r, mod.rms != 0, mod, [&](int k, int c) { return mod_chunk_global(mod, k, u, c); });
      }
    }
    rotate64<G>(v, ls);

    unsigned abits = __float_as_uint(absmax64(v));
#pragma unroll
    for (int off = 1; off < 32; off <<= 1)
      if (off < segw) abits = max(abits, __shfl_xor_sync(0xffffffffu, abits, off));
    const unsigned long long tag = static_cast<unsigned long long>(it + 1) << 32;
    if (active && (t % segw) == 0) atomicMax(&s_amax[slot][lr], tag | abits);
    __syncthreads();
    if (!active) continue;

    const float amax_z = __uint_as_float(static_cast<unsigned>(s_amax[slot][lr] & 0xffffffffull));
    // X_rot = z * 2^-n exactly, so max |X_rot| = amax_z * 2^-n.
    const float s = __fdiv_rn(amax_z * C::kInvScale, 127.0f);
    if (t == 0) scales[row] = s;
    const float d = held_divisor<G>(s, ls.flip);
    const bool zero_row = (s == 0.0f);
    const bool tiny_row = !zero_row && s < kMinNormal;
    const float rcp = (zero_row || tiny_row) ? 0.0f : __frcp_rn(d);

#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int u = in_unit_grouped<G>(gi, li, j);
      if (u >= units) continue;
      const int uo = out_unit<G>(u, gi, li, j);
      float qr[16];
      quantize_unit<G>(v[j], j, d, rcp, zero_row, tiny_row, qr);
      if (OUT == kPackI8) {
        int8_t* dst = static_cast<int8_t*>(out_codes) + row * static_cast<int64_t>(K) + 16 * uo;
        *reinterpret_cast<uint4*>(dst) = codes_i8(qr);
      } else {
        __half* dst = static_cast<__half*>(out_codes) + row * static_cast<int64_t>(K) + 16 * uo;
        uint4 lo, hi;
        codes_f16(qr, lo, hi);
        reinterpret_cast<uint4*>(dst)[0] = lo;
        reinterpret_cast<uint4*>(dst)[1] = hi;
      }
    }
  }
}

// ---- pack_tma_kernel: TMA-fed persistent pipeline ----------------------------

constexpr int kTmaMaxStages = 4;

struct PackTmaParams {
  CUtensorMap tmap;     // X as [M][L][E] elements (E per 128-B line), box {E, Lb, rbox}, 128-B swizzle
  void* out;            // codes [M, K], int8 or binary16
  float* scales;        // [M]
  float in_scale;       // input scale applied before the rotation (1 = none)
  ModPrologue mod;      // modulation prologue (kProModulate)
  int64_t M;
  int64_t nblocks;      // ceil(M / R)
  int K;
  int R;                // rows per block
  int tpr;              // threads per row
  int L;                // 128-byte lines per row
  int Lb;               // lines per TMA box
  int rbox;             // rows per TMA box: R when Lb == L (one box per block), else 1
  int nstages;
  uint32_t stage_bytes; // R * L * 128 rounded up to 1024
  // Separate code buffers: the codes of a block go to one of two buffers of
  // out_bytes (R * K * code size, rounded up to 1024) instead of over its
  // input stage, so that the stage is refilled as soon as every thread holds
  // its inputs (at the row-norm barrier, or the row-maximum barrier).
  int sep_out;
  uint32_t out_bytes;
};

// Shared memory (base aligned to 1024 B):
//   [nstages][stage_bytes]  input blocks, 128-byte swizzled lines; once a
//                           block is in registers its codes are written over
//                           it (natural layout) and bulk-copied out
//   [2][out_bytes]          (sep_out) the code buffers instead, used in turn
//   [kTmaMaxStages] u64     "stage full" barriers
//   [2][R] u64              tagged row absmax
//   [R][segments] f32       partial sums of squares (RMS norm)
//   int                     abort flag
//   [tpr][kModStride] 16 B  modulation vector chunks (kProModulate; 16-byte aligned)
template <int G, typename TIn, int OUT, int PRO>
__global__ void __launch_bounds__(kMaxThreads)
pack_tma_kernel(const __grid_constant__ PackTmaParams p) {
  using C = Geo<G>;
  constexpr int ESZ = static_cast<int>(sizeof(TIn));
  constexpr int OSZ = (OUT == kPackI8) ? 1 : 2;
  constexpr int CPU = InTraits<TIn>::kChunksPerUnit;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* in_base = smem;
  uint8_t* out_base = smem + static_cast<size_t>(p.nstages) * p.stage_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(out_base + (p.sep_out ? 2 * static_cast<size_t>(p.out_bytes) : 0));
  unsigned long long* s_amax = reinterpret_cast<unsigned long long*>(full + kTmaMaxStages);
  // [R][segments per row]: partial sums of squares of the lane segments
  float* s_sumsq = reinterpret_cast<float*>(s_amax + 2 * p.R);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(s_sumsq + p.R * row_segments(p.tpr));
  float4* s_vec = reinterpret_cast<float4*>((reinterpret_cast<uintptr_t>(abort_flag) + 4 + 15) & ~uintptr_t(15));
  int* err = &g_pack_error;

  const int tid = threadIdx.x;
  const int K = p.K;
  const int R = p.R;
  const int tpr = p.tpr;
  const int lr = tid / tpr;
  const int t = tid - lr * tpr;
  const int units = K >> 4;
  const int gi = t / C::kTPG;
  const int li = t - gi * C::kTPG;
  const bool in_cta_row = lr < R;
  const int lr_read = in_cta_row ? lr : 0;  // padding threads read row 0 and store nothing
  const int S = p.nstages;
  float4* s_mod = s_vec + t * kModStride;  // kProModulate: this column's vector chunks

  // units of this thread: round-robin over the row for G <= 16, the group's top
  // digit for G >= 64
  int u_of[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) u_of[j] = (G <= 16) ? t + tpr * j : in_unit_grouped<G>(gi, li, j);

  pdl_launch_dependents();  // the next kernel may set itself up; it waits for this one before reading
  for (int i = tid; i < 2 * R; i += blockDim.x) s_amax[i] = 0ull;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&p.tmap);
  }
  if (PRO == kProModulate && lr == 0) {
    // the first row's threads stage the vector values of their units, once
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        const float* base = (k == 0) ? p.mod.weight : (k == 1) ? p.mod.scale : p.mod.shift;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (base && u_of[j] < units) s_mod[mod_slot(k, j, c)] = mod_chunk_global(p.mod, k, u_of[j], c);
      }
  }
  __syncthreads();

  const uint64_t pol_in = l2_policy_evict_first();
  const float in_scale = p.in_scale;
  const uint32_t block_bytes = static_cast<uint32_t>(R) * static_cast<uint32_t>(p.L) * 128u;
  // Thread 0 only: load block `blk` into stage `stage`.
  auto issue = [&](int64_t blk, int stage) {
    uint8_t* dst = in_base + static_cast<size_t>(stage) * p.stage_bytes;
    const int64_t row0 = blk * R;
    if (p.Lb == p.L) {  // one box holds the whole block
      mbar_arrive_expect_tx(&full[stage], block_bytes);  // rows past M are zero-filled and still counted
      tma_load_3d(dst, &p.tmap, &full[stage], 0, 0, static_cast<int32_t>(row0), pol_in);
    } else {
      const int64_t rem = p.M - row0;
      const int rows = rem < R ? static_cast<int>(rem) : R;
      mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(rows) * p.L * 128u);
      for (int r = 0; r < rows; ++r)
        for (int l0 = 0; l0 < p.L; l0 += p.Lb)
          tma_load_3d(dst + (static_cast<size_t>(r) * p.L + l0) * 128, &p.tmap, &full[stage], 0, l0,
                      static_cast<int32_t>(row0 + r), pol_in);
    }
  };

  const LaneSigns<G> ls = lane_signs<G>(li);
  const int seg = tpr & -tpr;
  const int segw = seg < 32 ? seg : 32;

  const int64_t stride = gridDim.x;
  int64_t n_issued = 0;  // thread 0: blocks issued (block i of this CTA goes to stage i % S)
  if (tid == 0)
    for (int s = 0; s < S; ++s)
      if (blockIdx.x + s * stride < p.nblocks) { issue(blockIdx.x + s * stride, s); ++n_issued; }

  // thread 0, sep_out: refill the stage of the current block with the block
  // S iterations ahead (every thread holds its inputs)
  auto refill = [&](int64_t blk, int stage) {
    const int64_t nb = blk + S * stride;
    if (nb < p.nblocks) {
      issue(nb, stage);
      ++n_issued;
    }
  };

  int it = 0;
  bool aborted = false;
  for (int64_t blk = blockIdx.x; blk < p.nblocks; blk += stride, ++it) {
    const int stage = it % S;
    const uint32_t phase = static_cast<uint32_t>((it / S) & 1);
    const bool landed = mbar_wait(&full[stage], phase, abort_flag, err);

    const int64_t row = blk * R + lr;
    const bool active = in_cta_row && row < p.M;
    uint8_t* sbuf = in_base + static_cast<size_t>(stage) * p.stage_bytes;

    float v[4][16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int u = u_of[j];
      uint4 c[CPU];
      if (u < units) {
#pragma unroll
        for (int k = 0; k < CPU; ++k) {
          // byte offset in the block, then the 128-byte swizzle of TMA
          const uint32_t o = static_cast<uint32_t>((lr_read * K + 16 * u) * ESZ + 16 * k);
          const uint32_t line = o >> 7;
          const uint32_t phys = (line << 7) | ((((o >> 4) & 7u) ^ (line & 7u)) << 4);
          c[k] = *reinterpret_cast<const uint4*>(sbuf + phys);
        }
      } else {
#pragma unroll
        for (int k = 0; k < CPU; ++k) c[k] = make_uint4(0u, 0u, 0u, 0u);
      }
      unit_to_f32<TIn>(c, v[j]);
      prologue_unit<PRO>(v[j]);
      if (in_scale != 1.0f) scale_unit(v[j], in_scale);
    }
    const int slot = it & 1;
    bool refilled = false;
    if (PRO == kProModulate) {
      float r = 1.0f;
      if (p.mod.rms) {
        // one slot per lane segment (the previous block's reads ended before
        // the barrier that follows its row maximum)
        const int nseg = tpr / segw;
        const float ss = row_sumsq_part(v, segw);
        if (active && (t % segw) == 0) s_sumsq[lr * nseg + t / segw] = ss;
        if (__syncthreads_or(!landed)) { aborted = true; break; }
        if (p.sep_out && tid == 0) refill(blk, stage);
        refilled = p.sep_out;
        r = rms_factor(row_sumsq(s_sumsq + lr_read * nseg, nseg), K, p.mod.eps);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (active && u_of[j] < units)
          modulate_unit(v[j], r, p.mod.rms != 0, p.mod,
                        [&](int k, int c) { return s_mod[mod_slot(k, j, c)]; });
    }
    rotate64<G>(v, ls);

    unsigned abits = __float_as_uint(absmax64(v));
#pragma unroll
    for (int off = 1; off < 32; off <<= 1)
      if (off < segw) abits = max(abits, __shfl_xor_sync(0xffffffffu, abits, off));
    const unsigned long long tag = static_cast<unsigned long long>(it + 1) << 32;
    if (active && (t % segw) == 0) atomicMax(&s_amax[slot * R + lr], tag | abits);
    // sep_out: the code buffer of this block was last read by the store two
    // blocks back (one bulk group per block)
    if (p.sep_out && tid == 0) bulk_wait_read<1>();
    // every thread has its inputs in registers past this barrier, so the
    // codes may overwrite the stage
    if (__syncthreads_or(!landed)) { aborted = true; break; }
    if (p.sep_out && !refilled && tid == 0) refill(blk, stage);
    uint8_t* obuf = p.sep_out ? out_base + static_cast<size_t>(it & 1) * p.out_bytes : sbuf;

    if (active) {
      const float amax_z = __uint_as_float(static_cast<unsigned>(s_amax[slot * R + lr] & 0xffffffffull));
      // X_rot = z * 2^-n exactly, so max |X_rot| = amax_z * 2^-n.
      const float s = __fdiv_rn(amax_z * C::kInvScale, 127.0f);
      if (t == 0) p.scales[row] = s;
      const float d = held_divisor<G>(s, ls.flip);
      const bool zero_row = (s == 0.0f);
      const bool tiny_row = !zero_row && s < kMinNormal;
      const float rcp = (zero_row || tiny_row) ? 0.0f : __frcp_rn(d);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int u = u_of[j];
        if (u >= units) continue;
        const int uo = out_unit<G>(u, gi, li, j);
        float qr[16];
        quantize_unit<G>(v[j], j, d, rcp, zero_row, tiny_row, qr);
        uint8_t* dst = obuf + static_cast<size_t>(lr * K + 16 * uo) * OSZ;
        if (OUT == kPackI8) {
          *reinterpret_cast<uint4*>(dst) = codes_i8(qr);
        } else {
          uint4 lo, hi;
          codes_f16(qr, lo, hi);
          reinterpret_cast<uint4*>(dst)[0] = lo;
          reinterpret_cast<uint4*>(dst)[1] = hi;
        }
      }
    }
    fence_proxy_async_smem();  // make the codes visible to the bulk copy
    __syncthreads();
    if (tid == 0) {
      const int64_t rem = p.M - blk * R;
      const int64_t rows = rem < R ? rem : R;
      uint8_t* gdst = static_cast<uint8_t*>(p.out) + static_cast<size_t>(blk * R) * K * OSZ;
      bulk_store(gdst, obuf, static_cast<uint32_t>(rows * K * OSZ));
      bulk_commit();
      if (!p.sep_out && blk + S * stride < p.nblocks) {
        // refill this stage once the store has read the codes out of it
        bulk_wait_read<0>();
        refill(blk, stage);
      }
    }
  }
  if (tid == 0) {
    bulk_wait_all();
    if (aborted) {
      // no copy may land after the CTA exits: wait (bounded) for the blocks
      // that were issued but not consumed
      for (int64_t i = it; i < n_issued; ++i)
        mbar_wait(&full[i % S], static_cast<uint32_t>((i / S) & 1), nullptr, err);
    }
  }
}

// ---- launchers ----------------------------------------------------------------

int gcd_int(int a, int b) { while (b) { int t = a % b; a = b; b = t; } return a; }

// Raise a kernel's dynamic shared-memory limit once per device (and size).
// `configured` is that kernel's own record of the limit set on each device.
std::mutex g_smem_mu;

template <typename Kern>
int ensure_smem(Kern kern, size_t smem, size_t (&configured)[64]) {
  std::mutex& mu = g_smem_mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_cuda_error(e);
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64 || smem > configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return set_cuda_error(e);
    if (dev >= 0 && dev < 64) configured[dev] = smem;
  }
  return CONVROT_OK;
}

template <int G, typename TIn, int OUT, int PRO>
int launch_pack_cpasync(const void* X, int64_t M, int K, float in_scale, const ModPrologue& mod, void* out,
                        float* scales, cudaStream_t stream) {
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
  auto kern = pack_kernel<G, TIn, OUT, PRO>;
  static size_t configured[64] = {};
  if (int st = ensure_smem(kern, smem, configured)) return st;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
  if (e != cudaSuccess) return set_cuda_error(e);
  if (per_sm < 1) per_sm = 1;
  const int64_t nblocks = (M + rpc - 1) / rpc;
  const int64_t grid = std::min<int64_t>(nblocks, static_cast<int64_t>(per_sm) * device_sm_count());
  kern<<<static_cast<unsigned>(grid), threads, smem, stream>>>(
      static_cast<const TIn*>(X), M, K, tpr, rpc, nblocks, two_stage, in_scale, mod, out, scales);
  return check_launch();
}

constexpr size_t kSmemPerCtaMax = 227 * 1024;
constexpr uint32_t kTargetBlockBytes = 24 * 1024;  // input bytes of one block
constexpr int kStages = 2;                          // blocks in flight per CTA
constexpr int kVecSmemMaxK = 4096;                  // longest rows whose modulation vectors are staged
// The modulated pack stages the modulation vectors once per CTA, so it takes
// larger blocks (more rows share them) in one stage, refilled at the row-norm
// barrier (its codes have buffers of their own). Measured on the DiT input
// (M = 4608, K = 3072, G = 256): 36.6 us against 43.9 us with the codes
// written over the stage and 40-47 us with 24 KB blocks; the plain pack is
// faster with its codes over the stage (more CTAs fit per SM).
constexpr uint32_t kModTargetBlockBytes = 48 * 1024;
constexpr int kModStages = 1;

// Shape of the TMA path for rows of K elements, or false when it does not apply.
// `extra`: shared-memory bytes the kernel needs besides the stages and its
// bookkeeping (the staged modulation vectors).
// `block_target`, `max_stages`: the input bytes of one block and the blocks
// in flight per CTA to aim for.
template <typename TIn, int OUT>
bool plan_tma(int K, PackTmaParams& p, int& threads, size_t& smem, size_t extra = 0,
              uint32_t block_target = kTargetBlockBytes, int max_stages = kStages, bool sep_out = false) {
  constexpr int ESZ = static_cast<int>(sizeof(TIn));
  const int64_t row_in = static_cast<int64_t>(K) * ESZ;
  if (row_in % 128 != 0) return false;
  const int L = static_cast<int>(row_in / 128);
  const int tpr = (K + 63) / 64;
  if (tpr > kMaxThreads) return false;
  int R, Lb, rbox;
  if (L <= 256) {
    R = static_cast<int>(block_target / row_in);
    R = std::max(1, std::min(R, std::min(256, kMaxThreads / tpr)));
    Lb = L;
    rbox = R;
  } else {
    // one row per block in boxes of Lb lines; every box starts on a 1024-byte
    // boundary of the swizzle pattern
    if (L % 8 != 0) return false;
    Lb = 0;
    for (int d = 256; d >= 8; d -= 8)
      if (L % d == 0) { Lb = d; break; }
    if (Lb == 0) return false;
    R = 1;
    rbox = 1;
  }
  const uint32_t stage_bytes = static_cast<uint32_t>(((static_cast<int64_t>(R) * L * 128 + 1023) / 1024) * 1024);
  const size_t misc = 1024 + kTmaMaxStages * 8 + static_cast<size_t>(R) * (16 + 4 * row_segments(tpr)) + 16 + extra;
  constexpr int OSZ = (OUT == kPackI8) ? 1 : 2;
  const uint32_t out_bytes =
      sep_out ? static_cast<uint32_t>(((static_cast<int64_t>(R) * K * OSZ + 1023) / 1024) * 1024) : 0u;
  const size_t fixed = misc + 2 * static_cast<size_t>(out_bytes);
  int S = max_stages;
  while (S > 1 && fixed + static_cast<size_t>(S) * stage_bytes > kSmemPerCtaMax) --S;
  smem = fixed + static_cast<size_t>(S) * stage_bytes;
  if (smem > kSmemPerCtaMax) return false;
  p.K = K;
  p.R = R;
  p.tpr = tpr;
  p.L = L;
  p.Lb = Lb;
  p.rbox = rbox;
  p.nstages = S;
  p.stage_bytes = stage_bytes;
  p.sep_out = sep_out ? 1 : 0;
  p.out_bytes = out_bytes;
  threads = ((R * tpr + 31) / 32) * 32;
  return true;
}

template <int G, typename TIn, int OUT, int PRO>
int launch_pack_t(const void* X, int64_t M, int K, float in_scale, const ModPrologue& mod, void* out,
                  float* scales, cudaStream_t stream) {
  PackTmaParams p;
  memset(&p, 0, sizeof(p));
  int threads = 0;
  size_t smem = 0;
  // the modulated pack keeps the modulation vectors in shared memory (48
  // 16-byte chunks and one of padding per thread of a row); rows longer than kVecSmemMaxK
  // features take the general kernel, which reads them from global memory
  if (PRO == kProModulate && K > kVecSmemMaxK)
    return launch_pack_cpasync<G, TIn, OUT, PRO>(X, M, K, in_scale, mod, out, scales, stream);
  const bool modulated = (PRO == kProModulate);
  const size_t extra = modulated ? static_cast<size_t>(kModStride * 16) * ((K + 63) / 64) + 16 : 0;
  if (!plan_tma<TIn, OUT>(K, p, threads, smem, extra, modulated ? kModTargetBlockBytes : kTargetBlockBytes,
                          modulated ? kModStages : kStages, modulated))
    return launch_pack_cpasync<G, TIn, OUT, PRO>(X, M, K, in_scale, mod, out, scales, stream);

  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return set_cuda_error(cudaErrorNotSupported);
  constexpr int E = 128 / static_cast<int>(sizeof(TIn));
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(E), static_cast<cuuint64_t>(p.L),
                              static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(K) * sizeof(TIn)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(E), static_cast<cuuint32_t>(p.Lb),
                             static_cast<cuuint32_t>(p.rbox)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt =
      (sizeof(TIn) == 4) ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = enc(&p.tmap, dt, 3, const_cast<void*>(X), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_cuda_error(cudaErrorInvalidValue);
  p.out = out;
  p.scales = scales;
  p.in_scale = in_scale;
  p.mod = mod;
  p.M = M;
  p.nblocks = (M + p.R - 1) / p.R;

  auto kern = pack_tma_kernel<G, TIn, OUT, PRO>;
  static size_t configured[64] = {};
  if (int st = ensure_smem(kern, smem, configured)) return st;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
  if (e != cudaSuccess) return set_cuda_error(e);
  if (per_sm < 1) return set_cuda_error(cudaErrorInvalidConfiguration);
  const int64_t grid = std::min<int64_t>(p.nblocks, static_cast<int64_t>(per_sm) * device_sm_count());
  kern<<<static_cast<unsigned>(grid), threads, smem, stream>>>(p);
  return check_launch();
}

template <typename TIn, int OUT, int PRO = kProNone>
int dispatch_group(const void* X, int64_t M, int K, int G, float a, void* out, float* scales, cudaStream_t s,
                   const ModPrologue& mod = ModPrologue{nullptr, nullptr, nullptr, 0.0f, 0}) {
  switch (G) {
    case 1: return launch_pack_t<1, TIn, OUT, PRO>(X, M, K, a, mod, out, scales, s);
    case 4: return launch_pack_t<4, TIn, OUT, PRO>(X, M, K, a, mod, out, scales, s);
    case 16: return launch_pack_t<16, TIn, OUT, PRO>(X, M, K, a, mod, out, scales, s);
    case 64: return launch_pack_t<64, TIn, OUT, PRO>(X, M, K, a, mod, out, scales, s);
    case 256: return launch_pack_t<256, TIn, OUT, PRO>(X, M, K, a, mod, out, scales, s);
    case 1024: return launch_pack_t<1024, TIn, OUT, PRO>(X, M, K, a, mod, out, scales, s);
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

// Packed signed 4-bit weights ("Packed INT4 convrot": low nibble first) to
// int8 and/or binary16 codes; 16 values (8 bytes) per thread.
__global__ void __launch_bounds__(256) w4_expand_kernel(const uint8_t* __restrict__ src, int64_t n8,
                                                        int8_t* __restrict__ q8, __half* __restrict__ q16) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const uint2 a = __ldcs(reinterpret_cast<const uint2*>(src) + i);
  const uint32_t w[2] = {a.x, a.y};
  int v[16];
#pragma unroll
  for (int k = 0; k < 2; ++k)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t byte = (w[k] >> (8 * b)) & 0xffu;
      const int lo = static_cast<int>(byte & 0xfu), hi = static_cast<int>(byte >> 4);
      v[8 * k + 2 * b] = lo >= 8 ? lo - 16 : lo;       // element 2j: low nibble
      v[8 * k + 2 * b + 1] = hi >= 8 ? hi - 16 : hi;   // element 2j+1: high nibble
    }
  if (q8) {
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      o[k] = (static_cast<uint32_t>(v[4 * k] & 0xff)) | (static_cast<uint32_t>(v[4 * k + 1] & 0xff) << 8) |
             (static_cast<uint32_t>(v[4 * k + 2] & 0xff) << 16) | (static_cast<uint32_t>(v[4 * k + 3] & 0xff) << 24);
    reinterpret_cast<uint4*>(q8)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (q16) {
    uint32_t h[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) h[k] = pack2_f16(v[2 * k], v[2 * k + 1]);
    uint4* d = reinterpret_cast<uint4*>(q16) + 2 * i;
    d[0] = make_uint4(h[0], h[1], h[2], h[3]);
    d[1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

}  // namespace

int launch_w4_expand(const uint8_t* src, int64_t n, int8_t* q8, __half* q16, cudaStream_t stream) {
  if (n == 0) return CONVROT_OK;
  const int64_t n8 = n / 16;  // 16 values = 8 packed bytes per thread
  const int64_t blocks = (n8 + 255) / 256;
  w4_expand_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(src, n8, q8, q16);
  return check_launch();
}

int launch_pack(const void* X, int x_dtype, int64_t M, int64_t K, int G,
                void* out_codes, int out_kind, float* scales, cudaStream_t stream, float in_scale) {
  if (M == 0) return CONVROT_OK;
  const int k = static_cast<int>(K);
  const float a = in_scale;
  if (x_dtype == CONVROT_F32) {
    return out_kind == kPackI8 ? dispatch_group<float, kPackI8>(X, M, k, G, a, out_codes, scales, stream)
                               : dispatch_group<float, kPackF16>(X, M, k, G, a, out_codes, scales, stream);
  }
  return out_kind == kPackI8 ? dispatch_group<__half, kPackI8>(X, M, k, G, a, out_codes, scales, stream)
                             : dispatch_group<__half, kPackF16>(X, M, k, G, a, out_codes, scales, stream);
}

int launch_pack_gelu(const float* X, int64_t M, int64_t K, int G, __half* out_codes, float* scales,
                     cudaStream_t stream) {
  if (M == 0) return CONVROT_OK;
  return dispatch_group<float, kPackF16, kProGelu>(X, M, static_cast<int>(K), G, 1.0f, out_codes, scales, stream);
}

int launch_pack_modulated(const float* X, int64_t M, int64_t K, int G, const float* weight, const float* scale,
                          const float* shift, int rms, float eps, void* out_codes, int out_kind, float* scales,
                          cudaStream_t stream) {
  if (M == 0) return CONVROT_OK;
  const ModPrologue mod{weight, scale, shift, eps, rms};
  const int k = static_cast<int>(K);
  return out_kind == kPackI8
             ? dispatch_group<float, kPackI8, kProModulate>(X, M, k, G, 1.0f, out_codes, scales, stream, mod)
             : dispatch_group<float, kPackF16, kProModulate>(X, M, k, G, 1.0f, out_codes, scales, stream, mod);
}

int read_and_clear_pack_error() {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_pack_error, sizeof(int));
  if (e != cudaSuccess) return set_cuda_error(e);
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_pack_error, &zero, sizeof(int));
    if (e != cudaSuccess) return set_cuda_error(e);
  }
  return v;
}

int launch_widen(const int8_t* src, __half* dst, int64_t n, cudaStream_t stream) {
  if (n == 0) return CONVROT_OK;
  const int64_t n16 = n / 16;
  const int64_t blocks = (n16 + 255) / 256;
  widen_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(src, dst, n16);
  return check_launch();
}

}  // namespace convrot
