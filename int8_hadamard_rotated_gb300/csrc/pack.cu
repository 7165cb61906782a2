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
// How it computes it. With S = diag(1,1,1,-1) and P the swap of entries 1
// and 2, the page's H4 factors as H4 = 1/2 P S (H2 (x) H2) S, where H2 (x) H2
// is the 4-point Walsh-Hadamard matrix. The Kronecker power therefore is
//     R_G = 2^-n  P_G S_G W_G S_G,
// with W_G the G-point Walsh-Hadamard matrix (radix-2 butterflies on the
// index bits, in any order), S_G the sign flip of every index whose count of
// base-4 digits equal to 3 is odd, and P_G the swap of the two bits of every
// base-4 digit of the index. The kernel applies the input signs, the
// butterflies, the output signs, and writes each result at its bit-swapped
// position; the 2^-n normalisation is folded into the divisor exactly.
//
// Data layout. A thread owns 64 elements of one row: four "units" of 16
// consecutive elements (index bits 0-3 in registers). For G >= 64 the four
// units are the four values of the group's top base-4 digit (registers); the
// digits between bit 4 and the top digit live on G/64 consecutive lanes
// (shuffles). A row is processed by ceil(K/64) threads of one CTA; the row
// absmax is a warp-segment shuffle reduction plus one shared-memory atomic
// per segment. Loads are 16-byte vectors (a unit is 64 B of fp32), stores are
// one 16-byte vector per unit (int8) or two (fp16 codes).
#include "common.cuh"

#include <algorithm>

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

__device__ __forceinline__ float4 ld_stream(const float4* p) { return __ldcs(p); }
__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }

// Load the 16 elements of one unit as fp32.
template <typename TIn>
__device__ __forceinline__ void load_unit(const TIn* src, float (&v)[16]);

template <>
__device__ __forceinline__ void load_unit<float>(const float* src, float (&v)[16]) {
  const float4* s = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float4 a = ld_stream(s + i);
    v[4 * i + 0] = a.x; v[4 * i + 1] = a.y; v[4 * i + 2] = a.z; v[4 * i + 3] = a.w;
  }
}

template <>
__device__ __forceinline__ void load_unit<__half>(const __half* src, float (&v)[16]) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint4 a = ld_stream(s + i);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __half2 h = *reinterpret_cast<const __half2*>(&w[k]);
      float2 f = __half22float2(h);
      v[8 * i + 2 * k] = f.x;
      v[8 * i + 2 * k + 1] = f.y;
    }
  }
}

__device__ __forceinline__ uint32_t pack4_s8(int q0, int q1, int q2, int q3) {
  const uint32_t lo = __byte_perm(q0, q1, 0x0040);
  const uint32_t hi = __byte_perm(q2, q3, 0x0040);
  return __byte_perm(lo, hi, 0x5410);
}

__device__ __forceinline__ uint32_t pack2_f16(int q0, int q1) {
  __half2 h = __halves2half2(__int2half_rn(q0), __int2half_rn(q1));
  return *reinterpret_cast<uint32_t*>(&h);
}

constexpr int kMaxThreads = 512;

// One CTA handles `rpc` rows with `tpr` threads each.
template <int G, typename TIn, int OUT>
__global__ void __launch_bounds__(kMaxThreads)
pack_kernel(const TIn* __restrict__ X, int64_t M, int K, int tpr, int rpc,
            void* __restrict__ out_codes, float* __restrict__ scales) {
  using C = Geo<G>;
  __shared__ unsigned s_amax[kMaxThreads];

  const int tid = threadIdx.x;
  const int lr = tid / tpr;                 // row within the CTA
  const int t = tid - lr * tpr;             // thread within the row
  const int64_t row = static_cast<int64_t>(blockIdx.x) * rpc + lr;
  const bool active = (lr < rpc) && (row < M);
  const int units = K >> 4;
  const int gi = t / C::kTPG;
  const int li = t - gi * C::kTPG;

  if (tid < rpc) s_amax[tid] = 0u;

  // ---- load: four units, all loads issued before any use -----------------
  float v[4][16];
  const TIn* xrow = X + row * static_cast<int64_t>(K);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int u = gi * 4 * C::kTPG + j * C::kTPG + li;
    if (active && u < units) {
      load_unit<TIn>(xrow + 16 * u, v[j]);
    } else {
#pragma unroll
      for (int p = 0; p < 16; ++p) v[j][p] = 0.0f;
    }
  }

  // ---- input signs (register digits; lane digits are folded below) ---------
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int p = 0; p < 16; ++p)
      if (static_sign<G>(j, p)) v[j][p] = -v[j][p];

  // ---- butterflies inside each unit ----------------------------------------
#pragma unroll
  for (int b = 0; b < C::kUnitBits; ++b) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int p = 0; p < 16; ++p)
        if (!((p >> b) & 1)) {
          const float a = v[j][p], c = v[j][p | (1 << b)];
          v[j][p] = a + c;
          v[j][p | (1 << b)] = a - c;
        }
  }
  // ---- butterflies across the four units (the group's top digit) ----------
  if (C::kUnitDigit) {
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (!((j >> b) & 1))
#pragma unroll
          for (int p = 0; p < 16; ++p) {
            const float a = v[j][p], c = v[j | (1 << b)][p];
            v[j][p] = a + c;
            v[j | (1 << b)][p] = a - c;
          }
  }
  // ---- butterflies across lanes --------------------------------------------
  // Each lane keeps its raw values; the true value is rho * v. The lane input
  // sign sigma(li) starts as rho; a butterfly on lane bit b turns
  //   true' = (bit ? -1 : 1) * true(self) + true(partner)
  // into v' = fma(v, s_b * rho(self) * rho(partner), v(partner)) with the new
  // residual rho'(self) = rho(partner).
  int rho_mask = 0;  // lane bits processed so far
  if (C::kLaneBits > 0) {
#pragma unroll
    for (int b = 0; b < C::kLaneBits; ++b) {
      const int pli = li ^ (1 << b);
      const int rs = lane_sign<G>(li ^ rho_mask);
      const int rp = lane_sign<G>(pli ^ rho_mask);
      const int sb = (li >> b) & 1;
      const float coef = ((sb ^ rs ^ rp) & 1) ? -1.0f : 1.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int p = 0; p < 16; ++p) {
          const float u = __shfl_xor_sync(0xffffffffu, v[j][p], 1 << b);
          v[j][p] = fmaf(v[j][p], coef, u);
        }
      rho_mask |= (1 << b);
    }
  }
  // residual lane sign of the held values, times the output lane sign
  const int lane_flip = (C::kLaneBits > 0) ? (lane_sign<G>(li ^ rho_mask) ^ lane_sign<G>(li)) : 0;

  // ---- row absmax ------------------------------------------------------------
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int p = 0; p < 16; ++p) amax = fmaxf(amax, fabsf(v[j][p]));
  unsigned abits = __float_as_uint(amax);
  // aligned lane segments of gcd(tpr, 32) lanes never straddle two rows
  const int seg = tpr & -tpr;  // lowest set bit; seg divides 32 when tpr % seg == 0
  const int segw = seg < 32 ? seg : 32;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1)
    if (off < segw) abits = max(abits, __shfl_xor_sync(0xffffffffu, abits, off));
  __syncthreads();  // s_amax initialised
  if (active && (t % segw) == 0) atomicMax(&s_amax[lr], abits);
  __syncthreads();
  if (!active) return;

  const float amax_z = __uint_as_float(s_amax[lr]);
  // X_rot = z * 2^-n exactly, so max |X_rot| = amax_z * 2^-n.
  const float s = __fdiv_rn(amax_z * C::kInvScale, 127.0f);
  if (t == 0) scales[row] = s;
  // z / (s * 2^n) equals X_rot / s as a real number, hence the same rounded quotient.
  float d = s * C::kScale;
  if (lane_flip) d = -d;
  const bool zero_row = (s == 0.0f);

  // ---- quantize and store -----------------------------------------------------
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int u = gi * 4 * C::kTPG + j * C::kTPG + li;
    if (u >= units) continue;
    int uo;
    if (G <= 16) uo = u;
    else if (G == 64) uo = gi * 4 + swap2(j);
    else if (G == 256) uo = gi * 16 + swap2(j) * 4 + swap2(li);
    else uo = gi * 64 + swap2(j) * 16 + swap_digit_bits4(li);
    int q[16];
#pragma unroll
    for (int p = 0; p < 16; ++p) {
      // output sign of the register digits (same function as the input sign)
      const float z = static_sign<G>(j, p) ? -v[j][p] : v[j][p];
      int qi = zero_row ? 0 : __float2int_rn(__fdiv_rn(z, d));
      qi = min(max(qi, -127), 127);
      q[out_pos<G>(p)] = qi;
    }
    if (OUT == kPackI8) {
      int8_t* dst = static_cast<int8_t*>(out_codes) + row * static_cast<int64_t>(K) + 16 * uo;
      uint4 w;
      w.x = pack4_s8(q[0], q[1], q[2], q[3]);
      w.y = pack4_s8(q[4], q[5], q[6], q[7]);
      w.z = pack4_s8(q[8], q[9], q[10], q[11]);
      w.w = pack4_s8(q[12], q[13], q[14], q[15]);
      *reinterpret_cast<uint4*>(dst) = w;
    } else {
      __half* dst = static_cast<__half*>(out_codes) + row * static_cast<int64_t>(K) + 16 * uo;
      uint4 w0, w1;
      w0.x = pack2_f16(q[0], q[1]);   w0.y = pack2_f16(q[2], q[3]);
      w0.z = pack2_f16(q[4], q[5]);   w0.w = pack2_f16(q[6], q[7]);
      w1.x = pack2_f16(q[8], q[9]);   w1.y = pack2_f16(q[10], q[11]);
      w1.z = pack2_f16(q[12], q[13]); w1.w = pack2_f16(q[14], q[15]);
      reinterpret_cast<uint4*>(dst)[0] = w0;
      reinterpret_cast<uint4*>(dst)[1] = w1;
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
  while (threads * 2 <= 256 && tpr * rpc * 2 <= kMaxThreads) {
    rpc *= 2;
    threads = ((tpr * rpc + 31) / 32) * 32;
  }
  const int64_t grid = (M + rpc - 1) / rpc;
  if (grid > 0x7fffffff) return CONVROT_ERR_UNSUPPORTED;
  pack_kernel<G, TIn, OUT><<<static_cast<unsigned>(grid), threads, 0, stream>>>(
      static_cast<const TIn*>(X), M, K, tpr, rpc, out, scales);
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
