// common.cuh -- device helpers shared by the convrot kernels (sm_103a).
//
// Thin inline-PTX wrappers for mbarriers, TMA tensor copies and the tcgen05
// tensor-memory / MMA instructions, the device-side sticky error word, and
// host-side launch helpers. Every spin-wait here is bounded: on giving up it
// records CONVROT_ERR_TIMEOUT in the error word and returns false, so a kernel
// can release what it holds and exit instead of hanging the GPU.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "../../include/convrot.h"

namespace convrot {

// ---------------------------------------------------------------------------
// device error word
// ---------------------------------------------------------------------------

// Record `code` in a sticky device error word (first error wins). The word
// itself lives in the translation unit of the kernel that waits.
__device__ __forceinline__ void record_error(int* word, int code) {
  atomicCAS(word, 0, code);
}

// Upper bound on a single mbarrier wait, in nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// shared-memory addresses and mbarriers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
               ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed. Returns false
// (after recording a timeout in *err_word) if it does not complete within
// limit_ns, or early if `*abort_flag` (shared; may be null) is set by
// another thread.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort_flag, int* err_word,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 63) {
      if (abort_flag && *abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        if (abort_flag) *abort_flag = 1;
        record_error(err_word, CONVROT_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// TMA (tensor-map bulk copies)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// 2-D tiled load global -> shared, completion counted on `bar` in bytes.
// x = innermost coordinate (elements), y = row coordinate.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, uint64_t* bar,
                                            int32_t x, int32_t y, uint64_t cache_hint) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(smem_u32(smem_dst)), "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(cache_hint)
      : "memory");
}

// 3-D tiled load global -> shared (coordinates innermost first).
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* tmap, uint64_t* bar,
                                            int32_t x, int32_t y, int32_t z, uint64_t cache_hint) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;"
      ::"r"(smem_u32(smem_dst)), "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(cache_hint)
      : "memory");
}

// 2-D tiled store shared -> global through a tensor map (elements outside the
// tensor are not written), tracked by the issuing thread's bulk-async groups.
__device__ __forceinline__ void tma_store_2d(const void* tmap, const void* smem_src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
               ::"l"(tmap), "r"(smem_u32(smem_src)), "r"(x), "r"(y) : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start
// launching (its own prologue), and, in that kernel, wait until every kernel
// it depends on has completed and its writes are visible.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prerequisites() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Barrier over `nthreads` threads (a multiple of 32) using hardware barrier `id` (1..15).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Barrier over `nthreads` threads that also returns whether `pred` holds on
// every one of them (the same answer for all).
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r) : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads) : "memory");
  return r != 0;
}

// gpu-scope flag words
__device__ __forceinline__ unsigned long long ld_acquire_gpu(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_gpu(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Untiled bulk copy shared -> global (both 16-byte aligned, bytes % 16 == 0),
// tracked by the issuing thread's bulk-async groups.
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               ::"l"(gdst), "r"(smem_u32(ssrc)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// L2 cache-policy hints for TMA loads (createpolicy.fractional, fraction 1.0).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// 32-bit global stores carrying an L2 cache-policy hint.
__device__ __forceinline__ void st_global_hint(float* ptr, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(ptr), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_global_hint(int32_t* ptr, int32_t v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.s32 [%0], %1, %2;" ::"l"(ptr), "r"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// thread-block clusters (CTA pairs)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Shared::cluster address of the variable at shared::cta address `addr` in
// the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive once on an mbarrier given by its shared::cluster address (any CTA of the cluster).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Barrier over every thread of every CTA in the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 2-D tiled load into this CTA's shared memory whose completion is counted on
// an mbarrier of either CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const void* tmap, uint32_t bar_cluster_addr,
                                                 int32_t x, int32_t y, uint64_t cache_hint) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(smem_u32(smem_dst)), "l"(tmap), "r"(x), "r"(y), "r"(bar_cluster_addr), "l"(cache_hint)
      : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation MMA
// ---------------------------------------------------------------------------

// Allocate `ncols` TMEM columns (power of two >= 32); the base address is
// written to *dst_smem. Executed by one full warp.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               ::"r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (fp16 inputs, fp32 accumulate).
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when all tcgen05.mma issued so far by this thread complete.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_u32(bar)) : "memory");
}

// CTA-pair forms: TMEM allocation by one warp in each CTA of the pair (the
// same columns in both), the MMA issued by one thread of the pair with A and
// B split between the two CTAs' shared memory, and commits that arrive on the
// mbarrier at the same offset in every CTA of `cta_mask`.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
               ::"r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma_f16_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
      ::"r"(smem_u32(bar)), "h"(cta_mask) : "memory");
}

// Each thread of the warp reads its TMEM lane (32 lanes from the warp's lane
// quarter) and 32 consecutive 32-bit columns starting at taddr.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored with the
// 128-byte swizzle (rows of 64 fp16 = 128 B, 8-row atoms of 1024 B):
//   bits  0-13 start address >> 4      bits 16-29 leading byte offset >> 4
//   bits 32-45 stride byte offset >> 4 bits 46-47 descriptor version (1)
//   bits 49-51 base offset (0: atoms 1024-B aligned)
//   bits 61-63 swizzle mode (2 = 128-byte swizzle)
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1u) << 16;                 // LBO (unused for swizzled K-major)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;         // SBO: 8 rows x 128 B
  d |= static_cast<uint64_t>(1u) << 46;                 // version
  d |= static_cast<uint64_t>(2u) << 61;                 // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (K-major), fp32 D.
//   bits 4-5 D format (1 = f32)   bits 7-9 A format (0 = f16)
//   bits 10-12 B format (0 = f16) bits 15/16 A/B major (0 = K)
//   bits 17-22 N >> 3             bits 24-28 M >> 4
__host__ __device__ constexpr uint32_t idesc_f16_f32(uint32_t M, uint32_t N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// ---------------------------------------------------------------------------
// activations (GEMM epilogues, the MLP repack)
// ---------------------------------------------------------------------------

// GELU 0.5 y (1 + erf(y / sqrt 2)) with erf from Abramowitz & Stegun,
// "Handbook of Mathematical Functions", formula 7.1.28 (Hastings):
//   erf(t) = 1 - 1 / (1 + a1 t + a2 t^2 + ... + a6 t^6)^16 + e(t), |e| <= 3e-7,
// for t >= 0. P = 1 + a1 t + ... is formed by Horner's rule in fp32, 1 / P
// by the hardware reciprocal (rcp.approx, relative error about 2^-23) and
// raised to the 16th power by squaring; for y < 0, 1 + erf(-t) = 1 / P^16
// directly (no cancellation), for y >= 0, 1 + erf(t) = 2 - 1 / P^16. The
// result stays within about 5e-7 |y| of the exact GELU. Two elements at a
// time, on lane-wise fp32 pairs (each lane rounded as the scalar operation).
__device__ __forceinline__ unsigned long long f32x2_pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f32x2_unpack(unsigned long long r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long f32x2_fma(unsigned long long a, unsigned long long b,
                                                        unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ unsigned long long f32x2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void gelu_as2(float& y0, float& y1) {
  const unsigned long long t = f32x2_mul(f32x2_pack(fabsf(y0), fabsf(y1)),
                                         f32x2_pack(0.70710678118654752f, 0.70710678118654752f));
  auto c = [](float v) { return f32x2_pack(v, v); };
  unsigned long long P = f32x2_fma(t, c(0.0000430638f), c(0.0002765672f));
  P = f32x2_fma(t, P, c(0.0001520143f));
  P = f32x2_fma(t, P, c(0.0092705272f));
  P = f32x2_fma(t, P, c(0.0422820123f));
  P = f32x2_fma(t, P, c(0.0705230784f));
  P = f32x2_fma(t, P, c(1.0f));
  float p0, p1;
  f32x2_unpack(P, p0, p1);
  unsigned long long r = f32x2_pack(rcp_approx(p0), rcp_approx(p1));
  r = f32x2_mul(r, r);  // ^2
  r = f32x2_mul(r, r);  // ^4
  r = f32x2_mul(r, r);  // ^8
  r = f32x2_mul(r, r);  // ^16
  float r0, r1;
  f32x2_unpack(r, r0, r1);
  const float e0 = (y0 >= 0.0f) ? 2.0f - r0 : r0;  // 1 + erf
  const float e1 = (y1 >= 0.0f) ? 2.0f - r1 : r1;
  f32x2_unpack(f32x2_mul(f32x2_mul(f32x2_pack(y0, y1), c(0.5f)), f32x2_pack(e0, e1)), y0, y1);
}

// silu(g) * u = g u / (1 + exp(-g)), with exp(-g) = 2^(-g log2 e) from the
// hardware base-2 exponential (ex2.approx) and a correctly rounded
// reciprocal: a relative error of a few 1e-7 for |g| up to ~10, the exact
// limits 0 (g -> -inf) and g u (g -> +inf).
__device__ __forceinline__ float silu_mul_fast(float g, float u) {
  float e;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-1.4426950408889634f * g));
  return g * __frcp_rn(1.0f + e) * u;
}

// ---------------------------------------------------------------------------
// host helpers
// ---------------------------------------------------------------------------

int set_cuda_error(cudaError_t e);   // records e for convrot_last_cuda_error
int check_launch();                  // cudaGetLastError -> status

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// G is 4^n with 1 <= G <= 1024 and divides K.
bool valid_group(int G, int64_t K);
// b rounded up to a multiple of 256.
size_t round256(size_t b);
// CONVROT_OK on an sm_103 device, else CONVROT_ERR_DEVICE.
int check_device();

// cuTensorMapEncodeTiled from the driver (looked up once), or null.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn get_encode_fn();

// Number of SMs of the current device (cached per device).
int device_sm_count();
// Whether the current device is sm_103 (cached per device).
bool device_is_sm103();

// ---------------------------------------------------------------------------
// kernel launchers (implemented in pack.cu / gemm.cu)
// ---------------------------------------------------------------------------

enum PackOut { kPackI8 = 0, kPackF16 = 1 };

// Rotate + quantize rows of X. out_codes is int8 (kPackI8) or fp16 (kPackF16).
// in_scale multiplies every element before the rotation (1 = the plain pack).
int launch_pack(const void* X, int x_dtype, int64_t M, int64_t K, int G,
                void* out_codes, int out_kind, float* scales, cudaStream_t stream, float in_scale = 1.0f);

// The same pack of fp32 rows into binary16 codes with GELU (gelu_as2) applied
// to every element as it is loaded (the MLP's activation, fused into its
// repack).
int launch_pack_gelu(const float* X, int64_t M, int64_t K, int G, __half* out_codes, float* scales,
                     cudaStream_t stream);

// The pack of fp32 rows with the modulation prologue applied first: each row
// divided by sqrt(mean(x^2) + eps) (rms != 0), times weight[k], then
// (x + x * scale[k]) + shift[k]; null vectors are skipped.
int launch_pack_modulated(const float* X, int64_t M, int64_t K, int G, const float* weight, const float* scale,
                          const float* shift, int rms, float eps, void* out_codes, int out_kind, float* scales,
                          cudaStream_t stream);

// Packed signed 4-bit codes (two per byte, low nibble first) -> int8 and/or
// binary16 codes, n elements, n % 16 == 0; either output may be null.
int launch_w4_expand(const uint8_t* src, int64_t n, int8_t* q8, __half* q16, cudaStream_t stream);

// int8 codes -> fp16 codes (exact), n elements, n % 16 == 0.
int launch_widen(const int8_t* src, __half* dst, int64_t n, cudaStream_t stream);

struct GemmLinear {
  const __half* w16;   // [N,K] fp16 weight codes, or null for packed 4-bit weights
  const float* s_w;    // [N] or null
  const float* bias;   // [N] or null
  void* out;           // [M,N] fp32 Y or int32 A
  int64_t N;
  const int32_t* kchunk;  // [ceil(N/128)] exact-chunk plan (64-wide K blocks per chunk) or null
  float in_scale = 1.0f;       // the activations were packed times this; Y is divided by it before the bias
  const uint8_t* w4 = nullptr;  // [N,K/2] packed signed 4-bit weights (low nibble first), when w16 is null
};

// The GEMM operand of a weight descriptor (binary16 codes or packed 4-bit
// weights) and the device bytes it spans.
inline const void* weight_codes(const convrot_weight& w) {
  return w.q16 ? static_cast<const void*>(w.q16) : static_cast<const void*>(w.q4);
}
inline size_t weight_code_bytes(const convrot_weight& w, int64_t K) {
  return w.q16 ? static_cast<size_t>(w.N) * K * 2 : static_cast<size_t>(w.N) * K / 2;
}
// A weight descriptor as one linear of a GEMM launch, writing `out`.
inline GemmLinear to_linear(const convrot_weight& w, void* out, float in_scale = 1.0f) {
  GemmLinear l{reinterpret_cast<const __half*>(w.q16), w.scale, w.bias, out, w.N, w.q16 ? w.kchunk : nullptr,
               in_scale};
  l.w4 = w.q16 ? nullptr : w.q4;
  return l;
}

// Exact-chunk plan of int8 weight codes (see convrot_weight_chunks).
int launch_chunk_plan(const int8_t* Q_w, int64_t N, int64_t K, int32_t* kchunk, cudaStream_t stream);

// Device words through which the CTA pairs of one GEMM launch hand partial
// sums of split tiles to each other (the balanced tail): CONVROT_GEMM_SYNC_BYTES
// of caller scratch, 16-byte aligned, not used by any other launch while the
// GEMM runs. Words the GEMM consumes are left zero for the next launch. With no
// words the GEMM takes whole tiles only.
struct GemmSync {
  unsigned long long* words = nullptr;
  size_t bytes = 0;
  // test of the timeout path (convrot_test_handover_timeout): a wait limit for
  // the launch (0: the normal kWaitLimitNs) and whether the tails of split
  // tiles wait for a hand-over value that no head publishes
  unsigned long long test_wait_ns = 0;
  bool test_unpublished_handover = false;
};

// The hand-over words at `base` (CONVROT_GEMM_SYNC_BYTES of workspace).
inline GemmSync sync_at(void* base) {
  return GemmSync{static_cast<unsigned long long*>(base), CONVROT_GEMM_SYNC_BYTES};
}

// out_j = epilogue(x16 . w16_j^T) for every linear j; raw_s32 selects int32 A.
int launch_gemm(const __half* x16, const float* s_x, int64_t M, int64_t K,
                const GemmLinear* lins, int n_lin, bool raw_s32, cudaStream_t stream,
                GemmSync sync = GemmSync());

// The same for linears with packed 4-bit weights (w4): the S8 x S4 GEMM, which
// reads the packed bytes. K % 64 == 0, K <= CONVROT_W4_MAX_K, N % 4 == 0
// unless raw_s32.
int launch_gemm_w4(const __half* x16, const float* s_x, int64_t M, int64_t K,
                   const GemmLinear* lins, int n_lin, bool raw_s32, cudaStream_t stream,
                   GemmSync sync = GemmSync(), bool gelu = false);

// Every linear of the list, binary16-weight and packed 4-bit ones in one
// launch each (in that order, on the same stream and hand-over words).
int launch_linears(const __half* x16, const float* s_x, int64_t M, int64_t K,
                   const GemmLinear* lins, int n_lin, bool raw_s32, cudaStream_t stream,
                   GemmSync sync = GemmSync());

// The GEMM with an activation applied to its output before the store:
// CONVROT_ACT_GELU (every linear), CONVROT_ACT_SWIGLU (lins[0] = gate,
// lins[1] = up, same N; h = silu(gate) * up written to lins[0].out), or
// CONVROT_ACT_NONE. N % 4 == 0, no input scale; packed 4-bit weights with
// GELU or none only.
int launch_gemm_act(const __half* x16, const float* s_x, int64_t M, int64_t K,
                    const GemmLinear* lins, int n_lin, int act, cudaStream_t stream,
                    GemmSync sync = GemmSync());

// Test of the GEMM epilogue's unscaling step (gemm.cu): for each of
// n_divisors divisors a and every significand of y = 1.m * 2^y_exp, the step
// against the IEEE division; adds the count of results that differ to
// *mismatches and lowers *first to the smallest (index << 32 | y bits) of them.
int launch_unscale_sweep(const float* divisors, int n_divisors, int y_exp, unsigned long long* mismatches,
                         unsigned long long* first, cudaStream_t stream);

// Activation rows per tile (256, 192 or 128) for a grouped launch (gemm.cu).
int pick_tile_rows(int64_t M, const GemmLinear* lins, int n_lin, int pairs, bool can_split);

// ---------------------------------------------------------------------------
// host-side checks and the grouped launch shared by the entry points (api.cu)
// ---------------------------------------------------------------------------

// n_weights in [1, CONVROT_MAX_LINEARS]; every non-empty descriptor has Y and
// exactly one of q16, q4.
int check_weight_list(const convrot_weight* weights, int n_weights);
// Alignment and aliasing of the weight descriptors against each other and
// against the activation-side arrays [in0, in0+n0) and [in1, in1+n1).
int check_weights(const convrot_weight* weights, int n_weights, int64_t M, int64_t K,
                  const void* in0, size_t n0, const void* in1, size_t n1);
// One grouped GEMM over the non-empty linears, on packed fp16 codes + s_x.
int launch_grouped(const __half* x16, const float* s_x, int64_t M, int64_t K,
                   const convrot_weight* weights, int n_weights, cudaStream_t s, float in_scale = 1.0f,
                   GemmSync sync = GemmSync());

}  // namespace convrot
