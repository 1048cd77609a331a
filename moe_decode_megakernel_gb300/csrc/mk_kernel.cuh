// mk_kernel.cuh -- the persistent decode megakernel for sm_103a.
//
// One CTA per SM, resident for the whole decode step ("Cohere: a decode
// megakernel for North Mini Code", section "What is a Megakernel?").  The
// CTA has four roles, fixed per warp:
//   warp 0      controller: copies the SM's task descriptors from global
//               memory into a small shared-memory ring ("The task
//               descriptor": the controller stays ahead of the workers);
//   warp 1      producer: turns each task into work items and streams the
//               task's weight rows / KV pages into a ring of 32 KB shared-
//               memory stages with bulk async copies (cp.async.bulk +
//               mbarrier complete_tx).  Weights never depend on the step's
//               activations, so the producer runs ahead across task
//               boundaries without waiting on any cross-SM barrier ("3.
//               Weight prefetch"); only the MoE claimers wait, for the
//               routing that decides which expert rows to stream;
//   warp 2      storer: publishes finished work items -- once the
//               consumers have arrived on an item's done barrier it adds 1,
//               with release semantics, to each counter the item signals
//               ("The threadblock shape": the storer signals the output
//               barriers), so no consumer waits on a release;
//   warps 3-10  consumers: wait on the item's cross-SM counters, compute
//               from the staged rows and write the outputs themselves
//               (decode outputs are a few hundred bytes per task, so they
//               need no store pipeline).
//
// Cross-SM synchronisation is a counter per dependency in global memory,
// zeroed before each step ("Barriers"): a producer task adds 1 with release
// semantics after its outputs are written; a waiting task spins with
// acquire loads until the count is reached.  Every wait has a time limit: on
// expiry the kernel records the failing barrier, every role drains its
// in-flight copies and returns, and the host sees MK_ERR_TIMEOUT.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mk_internal.h"

namespace mk {
namespace dev {

constexpr uint32_t ERR_TIMEOUT = 1, ERR_PAGE = 2, ERR_INDEX = 3, ERR_SMEM_ALIGN = 4, ERR_RING = 5, ERR_RANGE = 6;
constexpr uint32_t FULL = 0xffffffffu;
constexpr int kBarConsumers = 1;  // named barrier id of the consumer warps
constexpr int kConsumerThreads = 32 * kConsumerWarps;

// --------------------------------------------------------------- PTX glue
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ int64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return static_cast<int64_t>(t);
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_n(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity), "r"(200000u)
      : "memory");
  return ok != 0;
}
// 1-D bulk copy global -> this CTA's shared memory, completing on an mbarrier.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* b) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(b))
      : "memory");
}
// The same copy with an L2 cache policy (evict_first for data read once per step).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* b,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(b)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}
// Eight products of a weight chunk (8 bf16) with activations xa (elements
// 0..3) and xb (4..7), fp32: even elements into a, odd into b.  Two fp32
// FMAs per packed instruction (each rounded as fmaf).
__device__ __forceinline__ void ffma2(float& a, float& b, float wa, float wb, float xa, float xb) {
  asm("{\n .reg .b64 rw, rx, racc;\n mov.b64 rw, {%2, %3};\n mov.b64 rx, {%4, %5};\n mov.b64 racc, {%0, %1};\n"
      " fma.rn.f32x2 racc, rw, rx, racc;\n mov.b64 {%0, %1}, racc;\n}"
      : "+f"(a), "+f"(b)
      : "f"(wa), "f"(wb), "f"(xa), "f"(xb));
}
__device__ __forceinline__ void dot8_bf16(uint4 u, uint4 xa, uint4 xb, float& a, float& b) {
  ffma2(a, b, __uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(xa.x), __uint_as_float(xa.y));
  ffma2(a, b, __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u), __uint_as_float(xa.z), __uint_as_float(xa.w));
  ffma2(a, b, __uint_as_float(u.z << 16), __uint_as_float(u.z & 0xffff0000u), __uint_as_float(xb.x), __uint_as_float(xb.y));
  ffma2(a, b, __uint_as_float(u.w << 16), __uint_as_float(u.w & 0xffff0000u), __uint_as_float(xb.z), __uint_as_float(xb.w));
}
// Four E4M3 codes (bytes of c, lowest first) as two f16x2 words: lo holds
// bytes 0 and 1, hi bytes 2 and 3 (the lower byte in the lower half).  Every
// E4M3 value is exact in f16.
__device__ __forceinline__ void e4m3x4_f16(uint32_t c, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}"
      : "=r"(lo), "=r"(hi)
      : "r"(c));
}
// Four E2M1 codes (the low 16 bits of c; a byte holds two codes, the
// earlier element in its low nibble) as two f16x2 words: lo from the low
// byte, hi from the next.  Every E2M1 value is exact in f16.
__device__ __forceinline__ void e2m1x4_f16(uint32_t c, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b8 a, b;\n .reg .b32 t;\n cvt.u8.u32 a, %2;\n shr.b32 t, %2, 8;\n cvt.u8.u32 b, t;\n"
      " cvt.rn.f16x2.e2m1x2 %0, a;\n cvt.rn.f16x2.e2m1x2 %1, b;\n}"
      : "=r"(lo), "=r"(hi)
      : "r"(c));
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// the lower (sel 0x1010) or upper (0x3232) half of an f16x2 in both halves
__device__ __forceinline__ uint32_t half_bcast(uint32_t a, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %1, %2;" : "=r"(r) : "r"(a), "r"(sel));
  return r;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
// f16x2 of (a, b), a in the lower half, round to nearest even
__device__ __forceinline__ uint32_t f16x2_rn(float a, float b) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}
// the two halves of an f16x2 word as binary32 (exact)
__device__ __forceinline__ float2 f16x2_f32(uint32_t h) {
  float a, b;
  asm("{\n .reg .b16 x, y;\n mov.b32 {x, y}, %2;\n cvt.f32.f16 %0, x;\n cvt.f32.f16 %1, y;\n}"
      : "=f"(a), "=f"(b)
      : "r"(h));
  return make_float2(a, b);
}
// 2-D TMA tile load (coordinates: x = element along the inner dimension, y = row).
__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* b, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(b)), "l"(policy)
      : "memory");
}
// ---- tcgen05: 5th-generation tensor cores with accumulators in tensor memory
// TMEM columns of this CTA's accumulator (power of two, >= 32), allocated by
// one warp; the TMEM address is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T: BF16 operands (both K-major), fp32 accumulator.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T: 8-bit operands (kind::f8f6f4, the formats
// named by the instruction descriptor; one MMA takes K = 32, 32 bytes of each
// K-major row), fp32 accumulator.
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// One arrival on `b` once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint64_t* b) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(b))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 16 consecutive fp32 columns of this thread's TMEM lane (the warp's quarter
// of the lanes, as the warp's index in the CTA modulo 4 selects).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// Shared-memory matrix descriptor of a K-major operand tile written by TMA
// with the 128-byte swizzle: rows of 128 bytes (64 BF16 of K) in atoms of 8
// rows, 1024 bytes from one atom to the next along M/N; the tile starts on a
// 1024-byte boundary.  Moving along K within the 128-byte row adds the byte
// offset to the start address.
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4)   // start address, 16-byte units
         | ((uint64_t)1 << 16)                 // leading-dimension offset (unused when swizzled)
         | ((uint64_t)(1024 >> 4) << 32)       // stride-dimension offset: one 8-row atom
         | ((uint64_t)1 << 46)                 // descriptor version
         | ((uint64_t)2 << 61);                // 128-byte swizzle
}
// Instruction descriptor of kind::f16: fp32 D, BF16 A and B, both K-major, M x N.
__host__ __device__ constexpr uint32_t tc_idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
// Instruction descriptor of kind::f8f6f4: fp32 D, E4M3 A and B (format 0),
// both K-major, M x N.
__host__ __device__ constexpr uint32_t tc_idesc_e4m3(int m, int n) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void tma_2d_plain(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* b) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(b))
      : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
// D += A (16x16, row) * B (16x8, col): BF16 operands, fp32 accumulation.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_volatile(const uint32_t* p) {
  return *reinterpret_cast<const volatile uint32_t*>(p);
}
__device__ __forceinline__ void bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Named barrier with an OR over the threads' predicates: a uniform decision.
__device__ __forceinline__ bool bar_or(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " barrier.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void consumers_sync() { bar_sync(kBarConsumers, kConsumerThreads); }

// ------------------------------------------------------------ numerics
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float bf16_f(uint16_t u) { return __uint_as_float((uint32_t)u << 16); }
__device__ __forceinline__ uint16_t f_bf16(float f) {  // round to nearest even (finite inputs)
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7f800000u) == 0x7f800000u) return (uint16_t)((u >> 16) | ((u & 0xffffu) ? 0x40u : 0u));
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
// (a, b) as two BF16 pairs whose sum carries 16 mantissa bits: hi = bf16(x),
// lo = bf16(x - hi).  Two MMAs on hi and lo give fp32-level products.
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const uint16_t ah = f_bf16(a), bh = f_bf16(b);
  hi = (uint32_t)ah | ((uint32_t)bh << 16);
  lo = (uint32_t)f_bf16(a - bf16_f(ah)) | ((uint32_t)f_bf16(b - bf16_f(bh)) << 16);
}
// Four consecutive activations as BF16 hi values (at hi) and lo values (at
// lo): the operand rows of the tcgen05 items (8-byte stores).
__device__ __forceinline__ void store_hilo4(uint16_t* hi, uint16_t* lo, float4 v) {
  uint32_t h0, l0, h1, l1;
  split_bf16x2(v.x, v.y, h0, l0);
  split_bf16x2(v.z, v.w, h1, l1);
  *reinterpret_cast<uint2*>(hi) = make_uint2(h0, h1);
  *reinterpret_cast<uint2*>(lo) = make_uint2(l0, l1);
}
// E4M3 codes (1 sign, 4 exponent, 3 mantissa bits; largest finite 448).
// f_e4m3x2 rounds two floats to nearest even, saturating at +-448, a's code
// in the low byte; e4m3_f is exact.
__device__ __forceinline__ uint32_t f_e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}
__device__ __forceinline__ float e4m3_f(uint32_t code) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)(code & 0xffu)));
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"((unsigned short)(h2 & 0xffffu)));
  return f;
}
// The FP8 tensor-core operand of four consecutive activations (|v| <= 448):
// kTcF8Terms E4M3 words, term j at row0 + j * term_stride.  Term j codes the
// remainder the earlier terms leave, times 16^j: v = sum_j code_j 16^-j to
// within 2^-16 |v| where |v| >= 2^-6, 2^-22 below (E4M3 keeps 4 significant
// bits and leaves at most 1/16 of its input; the differences are exact, since
// a code is within a factor of two of its input).
__device__ __forceinline__ void store_e4m3_terms4(uint8_t* row0, int64_t term_stride, float4 v) {
  float r0 = v.x, r1 = v.y, r2 = v.z, r3 = v.w;
#pragma unroll
  for (int j = 0; j < kTcF8Terms; ++j) {
    const uint32_t word = f_e4m3x2(r0, r1) | (f_e4m3x2(r2, r3) << 16);
    *reinterpret_cast<uint32_t*>(row0 + j * term_stride) = word;
    r0 = (r0 - e4m3_f(word)) * 16.f;
    r1 = (r1 - e4m3_f(word >> 8)) * 16.f;
    r2 = (r2 - e4m3_f(word >> 16)) * 16.f;
    r3 = (r3 - e4m3_f(word >> 24)) * 16.f;
  }
}
// 2^k with max_abs 2^k in [64, 128) (1 for 0 or a non-finite max): the
// power-of-two scale that brings a row into the E4M3 terms' range exactly.
__device__ __forceinline__ int e4m3_row_exponent(float max_abs) {
  const uint32_t bits = __float_as_uint(max_abs);
  const int e = (int)((bits >> 23) & 0xffu) - 127;  // max_abs in [2^e, 2^(e+1)) for normal values
  if (max_abs == 0.f || e == 128) return 0;
  const int k = 6 - (e < -126 ? -126 : e);
  return k > 126 ? 126 : k;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(FULL, v, m);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, m));
  return v;
}


// ----------------------------------------------------- shared memory map
struct Hdr {
  uint64_t full[kStages], empty[kStages];
  uint64_t dfull[kDescRing], dempty[kDescRing];
  uint64_t wfull[kWorkRing], wempty[kWorkRing];
  uint64_t done[kWorkRing];  // consumers finished the item in this slot
  int32_t desc[kDescRing][32];
  int32_t work[kWorkRing][32];
  // FP8 expert stages: the fp32 scales of the stage's rows, copied with the
  // rows (same full barrier); up/gate stages hold gate scales then up scales
  alignas(16) float scl[kStages][kMaxStageRows];
  // tcgen05 items: the accumulator is complete / every MMA has finished; the
  // TMEM address of the accumulator
  uint64_t acc_full, tc_drain;
  uint32_t tmem_addr;
  volatile int32_t abort;
  int32_t pad[28];
};

// the longest activation row a GEMV reads: hidden, intermediate (down
// projection) or one KV group's attention output (O projection)
template <class S>
__host__ __device__ constexpr int xs_row() {
  return S::H > S::I ? (S::H > S::G * S::D ? S::H : S::G * S::D) : (S::I > S::G * S::D ? S::I : S::G * S::D);
}

// The MoE tile plan of a kernel mode's expert weights (BF16, FP8 or FP4 rows).
template <class S, int M>
__host__ __device__ constexpr MoePlan plan_of() {
  return M == kModeTcFp8 ? S::mptc8 : mode_tc(M) ? S::mptc : mode_fp4(M) ? S::mp4 : mode_fp8(M) ? S::mp8 : S::mp;
}
// the stage plan of an expert tile that runs as a GEMV: in the tensor-core
// builds the same tiles in GEMV stages (experts with at most kTB rows)
template <class S, int M>
__host__ __device__ constexpr MoePlan gemv_plan_of() {
  return M == kModeTcFp8 ? S::mptcg8 : M == kModeTc ? S::mptcg : plan_of<S, M>();
}

template <class S>
struct Scratch {
  float xs[kTB * xs_row<S>()];              // activation rows of one GEMV pass (tagged)
  float out[2][kTB * kMaxStageRows];        // dot products of one stage (double buffer)
  alignas(16) uint16_t qh[8][S::D + 8];     // the KV group's queries (tagged), pre-scaled, as
  alignas(16) uint16_t ql[8][S::D + 8];     // BF16 hi + lo; rows >= G zero, padded rows
  float wred[kConsumerWarps][8];            // per-warp page maxima / sums per head
  float wsum[kConsumerWarps][8];
  alignas(16) uint16_t ph[8][S::P + 8];     // probabilities of one page, BF16 hi part [head][token]
  alignas(16) uint16_t pl[8][S::P + 8];     // and lo part (rows padded: conflict-free)
  float am[S::G], al[S::G], aa[S::G];       // running max, sum, rescale per head
  float red[kConsumerWarps * 2];
  double rope_theta[S::D / 2];              // base^(-2i/D)
  float2 rope_cs[kTB][S::D / 2];            // (cos, sin) of the step's rotation, rows < kTB
  int32_t row_pos[kTB], row_page[kTB];      // the step's new position and its page, rows < kTB
  int32_t xtag[4], qtag[4];                 // what xs / qs hold
  int32_t flag;                             // a block-wide decision (the last router task)
  int32_t tk_id[kConsumerWarps][S::K];      // top-k of the row a warp works on
  uint32_t tk_key[kConsumerWarps][S::K];
  unsigned long long mask[S::E];            // rows routed to each expert (bit b)
  int32_t ids[kMaxBatch * S::K];            // this layer's routing (top-k / finalize)
  int32_t cnt[S::E], off[S::E + 1], act[S::E + 1];
};

template <class S>
constexpr size_t smem_bytes() {
  return (size_t)kStages * kStageBytes + sizeof(Hdr) + sizeof(Scratch<S>);
}
constexpr size_t kMaxSmemPerCta = 232448;  // 227 KB of dynamic shared memory per CTA

// ---------------------------------------------------------------- shapes
template <int H_, int NQ_, int NKV_, int D_, int E_, int K_, int I_, int P_>
struct Shape {
  static constexpr int H = H_, NQ = NQ_, NKV = NKV_, D = D_, E = E_, K = K_, I = I_, P = P_;
  static constexpr int G = NQ / NKV;
  static constexpr int QKV = (NQ + 2 * NKV) * D;
  static constexpr ShapeDims dims{H, NQ, NKV, D, E, K, I, P};
  static constexpr MoePlan mp = moe_plan(dims);
  static constexpr MoePlan mp8 = moe_plan8(dims);  // FP8 expert rows
  static constexpr MoePlan mp4 = moe_plan4(dims);  // FP4 expert rows
  static constexpr MoePlan mptc = moe_plan_tc(dims);  // tcgen05 GEMM tiles
  static constexpr MoePlan mptc8 = moe_plan_tc8(dims);  // the same over FP8 expert rows
  static constexpr MoePlan mptcg = moe_plan_tc_gemv(dims);    // those tiles as GEMV stages
  static constexpr MoePlan mptcg8 = moe_plan_tc8_gemv(dims);
  static_assert(gemv_plan_fits(mptcg) && gemv_plan_fits(mptcg8), "GEMV stages divide the tcgen05 tiles");
  static constexpr int SR_H = stage_rows(H), SR_O = stage_rows(G * D), SR_I = stage_rows(I);
  static_assert(H % 256 == 0 && (G * D) % 8 == 0 && I % 8 == 0, "row chunks");
  static_assert(D % 32 == 0 && 32 % G == 0 && (G * D) % 4 == 0, "attention lane maps");
  static_assert((G * D / 4) <= kConsumerThreads, "PV threads");
  static_assert(2 * P * D * 2 <= kStageBytes, "one KV page per stage");
  static_assert(G <= 8 && D % 64 == 0 && P % 16 == 0 && P <= 64, "MMA attention shape");
  static_assert(E <= 256 && K <= 32, "routing scratch");
};

struct Ctx {
  Hdr* hdr;
  uint8_t* stages;
  int sm;
  uint32_t st;  // stages issued (producer) / consumed (consumers)
  uint32_t wk;  // work items pushed / popped
  uint64_t stat[4];
};

// ----------------------------------------------------------- errors/waits
struct ErrWhere {  // what to report with an error: the task, its opcode and layer
  int32_t task, op, layer;
};
__device__ __forceinline__ ErrWhere where_of(const int32_t* d) { return {d[F_TASK], d[F_OP], d[F_LAYER]}; }
constexpr ErrWhere kNowhere{-1, -1, -1};

static __device__ __noinline__ void record_error(const Params& p, uint32_t code, int sm, ErrWhere at, int bar,
                                                 uint32_t seen, uint32_t tgt) {
  if (atomicCAS(p.err, 0u, code) == 0u) {
    p.err[1] = (uint32_t)sm;
    p.err[2] = (uint32_t)at.task;
    p.err[3] = (uint32_t)bar;
    p.err[4] = seen;
    p.err[5] = tgt;
    p.err[6] = (uint32_t)at.op;
    p.err[7] = (uint32_t)at.layer;
    __threadfence();
  }
}

static __device__ __forceinline__ bool aborted(const Ctx& c) { return c.hdr->abort != 0; }

// Waits for an mbarrier phase; false if the CTA is aborting or the watchdog fired.
// Waits inside the CTA get four times the limit of the cross-SM waits, so that
// when a dependency never arrives, the wait on it is the one recorded.
static __device__ __forceinline__ bool mbar_wait(const Params& p, Ctx& c, uint64_t* b, uint32_t parity) {
  if (mbar_try_wait(b, parity)) return true;
  const int64_t t0 = gtimer();
  for (;;) {
    if (mbar_try_wait(b, parity)) return true;
    if (aborted(c)) return false;
    if (ld_volatile(p.err) != 0) {
      c.hdr->abort = 1;
      return false;
    }
    if (gtimer() - t0 > 4 * p.watchdog_ns) {
      record_error(p, ERR_TIMEOUT, c.sm, kNowhere, -1, 0, 0);
      c.hdr->abort = 1;
      return false;
    }
  }
}

// Waits until counter `bar` reaches `tgt` (one thread).  "Barriers": spin with
// a short sleep; here with acquire loads and a time limit.
static __device__ __forceinline__ bool wait_counter(const Params& p, Ctx& c, int bar, uint32_t tgt, ErrWhere at) {
  if (bar < 0 || tgt == 0) return true;
  const uint32_t* a = p.bars + bar;
  if (ld_acquire(a) >= tgt) return true;
  const int64_t t0 = gtimer();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(20);
    if (ld_acquire(a) >= tgt) return true;
    if ((it & 31u) == 0) {
      if (aborted(c)) return false;
      if (ld_volatile(p.err) != 0) {
        c.hdr->abort = 1;
        return false;
      }
      if (gtimer() - t0 > p.watchdog_ns) {
        record_error(p, ERR_TIMEOUT, c.sm, at, bar, ld_volatile(a), tgt);
        c.hdr->abort = 1;
        return false;
      }
    }
  }
}

// Two waits at once (either may be absent: bar < 0 or tgt 0): both counters
// are read in every round.
static __device__ __forceinline__ bool wait_counters(const Params& p, Ctx& c, int b0, uint32_t t0, int b1,
                                                     uint32_t t1, ErrWhere at) {
  const bool n0 = b0 >= 0 && t0 > 0, n1 = b1 >= 0 && t1 > 0;
  if (!n0 && !n1) return true;
  if (!n0) return wait_counter(p, c, b1, t1, at);
  if (!n1) return wait_counter(p, c, b0, t0, at);
  const uint32_t* a0 = p.bars + b0;
  const uint32_t* a1 = p.bars + b1;
  int64_t ts = 0;
  for (uint32_t it = 0;; ++it) {
    const uint32_t v0 = ld_acquire(a0), v1 = ld_acquire(a1);
    if (v0 >= t0 && v1 >= t1) return true;
    if (it == 0) ts = gtimer();
    __nanosleep(20);
    if ((it & 31u) == 31u) {
      if (aborted(c)) return false;
      if (ld_volatile(p.err) != 0) {
        c.hdr->abort = 1;
        return false;
      }
      if (gtimer() - ts > p.watchdog_ns) {
        const bool first = v0 < t0;
        record_error(p, ERR_TIMEOUT, c.sm, at, first ? b0 : b1, first ? v0 : v1, first ? t0 : t1);
        c.hdr->abort = 1;
        return false;
      }
    }
  }
}

static __device__ __forceinline__ int slices_of(const Params& p, int seq) {
  return (seq + p.split_len - 1) / p.split_len;
}

// ======================================================================
// controller
// ======================================================================
static __device__ void controller(const Params& p, Ctx& c) {
  if ((threadIdx.x & 31) != 0) return;
  const int off = p.sched[2 * c.sm], n = p.sched[2 * c.sm + 1];
  Hdr* H = c.hdr;
  int i = 0;
  for (; i < n; ++i) {
    const int slot = i % kDescRing;
    if (i >= kDescRing && !mbar_wait(p, c, &H->dempty[slot], ((i / kDescRing) - 1) & 1)) break;
    mbar_expect_tx(&H->dfull[slot], 128);
    bulk_g2s(H->desc[slot], p.sched + off + 32 * i, 128, &H->dfull[slot]);
    p.prog[c.sm * 8 + 7] = (uint32_t)(i + 1);
  }
  if (i < n) {  // aborted: let the copies already issued land before returning
    for (int j = (i > kDescRing ? i - kDescRing : 0); j < i; ++j) {
      const int64_t t0 = gtimer();
      while (!mbar_try_wait(&H->dfull[j % kDescRing], (j / kDescRing) & 1) && gtimer() - t0 < p.watchdog_ns) {
      }
    }
  }
}

// ======================================================================
// producer
// ======================================================================
template <class S, int M>
struct Producer {
  // the lean builds: static claims and separate MoE drains only
  static constexpr bool kLean = mode_lean(M);
  const Params& p;
  Ctx c;
  // weights and KV pages are read once per step: streaming them with
  // evict_first keeps L2 for activations, counters and the kernel's code
  uint64_t stream_policy;

  __device__ __forceinline__ bool acquire_stage(int& slot) {
    slot = c.st % kStages;
    if (c.st >= (uint32_t)kStages) {
      const int64_t t0 = p.stats ? gtimer() : 0;
      const bool ok = mbar_wait(p, c, &c.hdr->empty[slot], ((c.st / kStages) - 1) & 1);
      if (p.stats) c.stat[0] += gtimer() - t0;
      return ok;
    }
    return true;
  }
  __device__ __forceinline__ uint8_t* stage(int slot) { return c.stages + (size_t)slot * kStageBytes; }

  __device__ __forceinline__ bool push(const int32_t* item) {
    const int slot = c.wk % kWorkRing;
    if (c.wk >= (uint32_t)kWorkRing) {
      const int64_t t0 = p.stats ? gtimer() : 0;
      const bool ok = mbar_wait(p, c, &c.hdr->wempty[slot], ((c.wk / kWorkRing) - 1) & 1);
      if (p.stats) c.stat[2] += gtimer() - t0;
      if (!ok) return false;
    }
    int32_t* dst = c.hdr->work[slot];
    for (int i = 0; i < 32; ++i) dst[i] = item[i];
    dst[F_SEQ] = (int32_t)c.wk;
    mbar_arrive(&c.hdr->wfull[slot]);
    ++c.wk;
    p.prog[c.sm * 8 + 4] = c.st;
    p.prog[c.sm * 8 + 5] = c.wk;
    return true;
  }

  // Waits until the consumers finished work item k of this SM (the storer
  // handed its slot back).  k is the latest item pushed or an earlier one,
  // so the slot's barrier is at most one phase short of it.
  __device__ __forceinline__ bool item_finished(uint32_t k) {
    const int64_t t0 = p.stats ? gtimer() : 0;
    const bool ok = mbar_wait(p, c, &c.hdr->wempty[k % kWorkRing], (k / kWorkRing) & 1);
    if (p.stats) c.stat[2] += gtimer() - t0;
    return ok;
  }

  // rows [row0, row0+nrows) of a [rows][K] matrix (row stride `ld` elements),
  // SR rows per stage
  __device__ __forceinline__ bool load_rows(const uint16_t* base, int64_t ld, int K, int row0, int nrows, int SR) {
    for (int s0 = 0; s0 < nrows; s0 += SR) {
      const int rs = min(SR, nrows - s0);
      int slot;
      if (!acquire_stage(slot)) return false;
      uint64_t* fb = &c.hdr->full[slot];
      uint8_t* dst = stage(slot);
      const uint32_t bytes = (uint32_t)rs * K * 2;
      mbar_expect_tx(fb, bytes);
      if (ld == K) {
        bulk_g2s_hint(dst, base + (int64_t)(row0 + s0) * K, bytes, fb, stream_policy);
      } else {
        for (int r = 0; r < rs; ++r)
          bulk_g2s_hint(dst + (size_t)r * K * 2, base + (int64_t)(row0 + s0 + r) * ld, K * 2, fb, stream_policy);
      }
      ++c.st;
    }
    return true;
  }

  __device__ __forceinline__ int dense_stages(int rows, int SR) { return (rows + SR - 1) / SR; }

  // A GEMV item with more activation rows than the consumers' cache holds
  // (kTB) is streamed once per kTB rows: the consumers load each pair of
  // rows once and run every stage against it (a repeat pass mostly reads
  // the rows from L2, where the previous pass left them).
  __device__ __forceinline__ int gemv_passes(int ntok) {
    if constexpr (M != kModeAnyBatch) return 1;  // the other modes' steps have at most kTB rows
    return ntok > kTB ? (ntok + kTB - 1) / kTB : 1;
  }

  // ---- tcgen05 items (kModeTc) ----
  // The k-blocks of one item: per stage the weight box(es) of the item's
  // kTcRows rows (a, at column ax + kTcK kb and row ay; an up/gate tile takes
  // its 64 gate and 64 up rows in blocks of 16, gate block j then up block j,
  // so that gate row i and up row i meet in one warp's TMEM lanes) and the
  // activation box (b, rows by .. by + tc_nb).  The weight boxes need no
  // input: they go out at once, as far as the ring reaches.  The activation
  // rows are written by other SMs, so their boxes are copied only after the
  // item's input counters are complete (then a proxy fence: the rows were
  // written by ordinary stores, the copy reads through the async proxy).
  // With a weight box of a_bytes < kTcABytes (a router task's rows), a stage
  // takes kps = tc_kblocks_per_stage(a_bytes) k-blocks: weight box j at
  // j * a_bytes, activation box j at kTcABytes + j * (its bytes).
  // FP8 expert tiles (kModeTcFp8) take k-blocks of kk = kTcK8 one-byte
  // weights and activation boxes of nb = tc_nb8 term rows: 128-byte rows as
  // for BF16, so the stage layout is the same.
  __device__ __forceinline__ bool tc_stages(const int32_t* it, const CUtensorMap* ta, int ax, int ay, bool updown,
                                            const CUtensorMap* tb, int bx, int by, int nkb,
                                            uint32_t a_bytes = kTcABytes, int kk = kTcK, int nb = 0) {
    if (nb == 0) nb = p.tc_nb;
    const uint32_t bbytes = (uint32_t)nb * kTcK * 2;
    const int kps = tc_kblocks_per_stage(a_bytes, nb);
    const int nst = (nkb + kps - 1) / kps;
    const uint32_t first = c.st;
    bool ready = false;
    auto issue_b = [&](uint32_t gs, int st) {
      for (int j = 0; j < kps && st * kps + j < nkb; ++j) {
        uint8_t* dst = stage(gs % kStages) + kTcABytes + j * bbytes;
        tma_2d_plain(dst, tb, bx + (st * kps + j) * kk, by, &c.hdr->full[gs % kStages]);
      }
    };
    auto wait_inputs = [&]() -> bool {
      const int64_t t0 = p.stats ? gtimer() : 0;
      const bool ok = wait_counters(p, c, it[F_WAIT0], (uint32_t)it[F_TGT0], it[F_WAIT1], (uint32_t)it[F_TGT1],
                                    where_of(it));
      if (p.stats) c.stat[1] += gtimer() - t0;
      if (!ok) return false;
      fence_proxy_async_global();
      for (uint32_t gs = first; gs < c.st; ++gs) issue_b(gs, (int)(gs - first));
      return true;
    };
    for (int st = 0; st < nst; ++st) {
      // the next slot would be one of this item's own stages, still without its activations
      if (!ready && c.st - first >= (uint32_t)kStages) {
        if (!wait_inputs()) return false;
        ready = true;
      }
      int slot;
      if (!acquire_stage(slot)) return false;
      uint64_t* fb = &c.hdr->full[slot];
      uint8_t* dst = stage(slot);
      const int nk = min(kps, nkb - st * kps);
      mbar_expect_tx(fb, (uint32_t)nk * (a_bytes + bbytes));
      for (int j = 0; j < nk; ++j) {
        const int x = ax + (st * kps + j) * kk;
        if (updown) {  // 16-row blocks: gate block q, then up block q
#pragma unroll
          for (int q = 0; q < kTcMoeRows / 32; ++q) {
            tma_2d(dst + j * a_bytes + (2 * q) * 2048, &p.tm_wg, x, ay + 16 * q, fb, stream_policy);
            tma_2d(dst + j * a_bytes + (2 * q + 1) * 2048, &p.tm_wu, x, ay + 16 * q, fb, stream_policy);
          }
        } else {
          tma_2d(dst + j * a_bytes, ta, x, ay, fb, stream_policy);
        }
      }
      if (ready) issue_b(c.st, st);
      ++c.st;
    }
    return ready || wait_inputs();
  }

  // A dense GEMM task as one tcgen05 item: its rows (<= kTcRows) of the
  // weight matrix against every activation row of the step.
  __device__ __forceinline__ bool tc_dense(const int32_t* d) {
    int32_t it[32];
    for (int i = 0; i < 32; ++i) it[i] = d[i];
    const int op = d[F_OP], l = d[F_LAYER], row0 = d[F_A0];
    const CUtensorMap* ta;
    const CUtensorMap* tb = &p.tm_xb;
    int ax = 0, ay, bx = 0, nkb = S::H / kTcK;
    // dense tiles copy only their own rows (the MMA's other rows are unused),
    // several k-blocks per stage
    uint32_t a_bytes = kTcDenseRows * kTcK * 2;
    switch (op) {
      case OP_QKV_PROJ: ta = &p.tm_wqkv; ay = l * S::QKV + row0; break;
      case OP_ROUTER_GEMM: ta = &p.tm_wr; ay = l * S::E + row0; a_bytes = kTcRouterRows * kTcK * 2; break;
      case OP_LM_HEAD: ta = &p.tm_wlm; ay = row0; break;
      default:  // OP_O_PROJ: the columns of KV group g
        ta = &p.tm_wo; ay = l * S::H + row0; ax = bx = d[F_A0 + 2] * S::G * S::D; tb = &p.tm_attnb;
        nkb = S::G * S::D / kTcK; break;
    }
    it[F_NSTAGE] = (nkb + tc_kblocks_per_stage(a_bytes, p.tc_nb) - 1) / tc_kblocks_per_stage(a_bytes, p.tc_nb);
    it[F_A0 + 13] = nkb;
    if (!push(it)) return false;
    return tc_stages(it, ta, ax, ay, false, tb, bx, 0, nkb, a_bytes);
  }

  __device__ __forceinline__ bool dense(const int32_t* d) {
    if constexpr (mode_tc(M)) return tc_dense(d);
    int32_t it[32];
    for (int i = 0; i < 32; ++i) it[i] = d[i];
    const int op = d[F_OP], l = d[F_LAYER], row0 = d[F_A0], rows = d[F_A0 + 1];
    const uint16_t* base;
    int64_t ld;
    int K, SR;
    switch (op) {
      case OP_QKV_PROJ: base = p.wqkv + (int64_t)l * S::QKV * S::H; ld = S::H; K = S::H; SR = S::SR_H; break;
      case OP_ROUTER_GEMM: base = p.wr + (int64_t)l * S::E * S::H; ld = S::H; K = S::H; SR = S::SR_H; break;
      case OP_LM_HEAD: base = p.wlm; ld = S::H; K = S::H; SR = S::SR_H; break;
      default:  // OP_O_PROJ: the columns of KV group g
        base = p.wo + (int64_t)l * S::H * S::NQ * S::D + (int64_t)d[F_A0 + 2] * S::G * S::D;
        ld = S::NQ * S::D; K = S::G * S::D; SR = S::SR_O; break;
    }
    const int passes = gemv_passes(p.B);
    it[F_NSTAGE] = dense_stages(rows, SR) * passes;
    if (!push(it)) return false;
    for (int ps = 0; ps < passes; ++ps)
      if (!load_rows(base, ld, K, row0, rows, SR)) return false;
    return true;
  }

  // KV pages as TMA tiles of (P tokens, 64 dims), swizzled: the K page of group
  // g at the stage's start, its V page after it
  __device__ __forceinline__ bool attn_pages(int l, int b, int g, int pf, int np) {
    constexpr int BOXES = S::D / 64, BOX_BYTES = S::P * 128;
    for (int k = 0; k < np; ++k) {
      int slot;
      if (!acquire_stage(slot)) return false;
      uint64_t* fb = &c.hdr->full[slot];
      uint8_t* dst = stage(slot);
      int page = -1;
      const int lp = pf + k;
      if (lp < p.max_pages) page = __ldg(p.block_tables + (int64_t)b * p.max_pages + lp);
      if (page < 0 || page >= p.num_pages) {
        record_error(p, ERR_PAGE, c.sm, kNowhere, lp, (uint32_t)page, (uint32_t)p.num_pages);
        mbar_arrive(&c.hdr->full[slot]);  // complete the stage without data
      } else {
        const int row = (int)((((int64_t)l * p.num_pages + page) * S::NKV + g) * S::P);
        mbar_expect_tx(fb, (uint32_t)(2 * BOXES * BOX_BYTES));
#pragma unroll
        for (int bx = 0; bx < BOXES; ++bx) {
          tma_2d(dst + bx * BOX_BYTES, &p.tm_k, 64 * bx, row, fb, stream_policy);
          tma_2d(dst + (BOXES + bx) * BOX_BYTES, &p.tm_v, 64 * bx, row, fb, stream_policy);
        }
      }
      ++c.st;
    }
    return true;
  }

  // one KV slice [t0, t1) of (b, g) as a work item plus its pages
  __device__ __forceinline__ bool attn_item(const int32_t* d, int l, int b, int g, int t0, int t1, int slot_idx, int wait_bar,
                            int wait_tgt, int sig) {
    int32_t it[32];
    for (int i = 0; i < 32; ++i) it[i] = d[i];
    it[F_OP] = W_ATTN;
    it[F_LAYER] = l;
    it[F_WAIT0] = wait_bar;
    it[F_TGT0] = wait_tgt;
    it[F_WAIT1] = -1;
    it[F_SIG0] = sig;
    it[F_SIG1] = -1;
    const int pf = t0 / S::P;
    const int np = t1 > t0 ? (t1 - 1) / S::P - pf + 1 : 0;
    it[F_A0] = b;
    it[F_A0 + 1] = g;
    it[F_A0 + 2] = t0;
    it[F_A0 + 3] = t1;
    it[F_A0 + 4] = pf;
    it[F_A0 + 5] = slot_idx;
    it[F_NSTAGE] = np;
    if (!push(it)) return false;
    return attn_pages(l, b, g, pf, np);
  }

  __device__ __forceinline__ bool attn_decode(const int32_t* d) {
    const int l = d[F_LAYER], b = d[F_A0], g = d[F_A0 + 1], j = d[F_A0 + 2];
    int t0 = 0, t1 = 0;
    if (b < p.B) {
      const int s = __ldg(p.seq_lens + b);
      const bool full = p.window == 0 || (l + 1) % p.full_period == 0;
      const int lo = full ? 0 : max(0, s - p.window);
      const int jj = lo / p.split_len + j;
      t0 = max(lo, jj * p.split_len);
      t1 = min(s, (jj + 1) * p.split_len);
      if (t1 < t0) t1 = t0;
    }
    return attn_item(d, l, b, g, t0, t1, j, d[F_WAIT0], d[F_TGT0], d[F_SIG0]);
  }

  // Claimer over the full-attention queue ("Task scheduler": ATTN_DRAIN
  // claims the next entry until the queue is empty).  The queue holds one
  // entry per (row b, KV group g, slice j), ordered (b, g, j); entry i is
  // located from the rows' slice counts, so the queue needs no storage.
  // Dynamic claims: a claimer holds at most one slice beyond the one its consumers work on:
  // after pushing slice i it claims the next slice only when the item before
  // i is finished (its pages then load while i runs).  Run-ahead would leave
  // the early claimers with a backlog of slices while the late ones find the
  // queue empty.
  __device__ __forceinline__ bool attn_drain(const int32_t* d) {
    const int l = d[F_LAYER];
    uint32_t* claim = p.bars + d[F_A0];
    // static claims: claimer ci of n takes the entries ci, ci + n, ...
    const int ci = d[F_A0 + 4];
    const uint32_t n_cl = (uint32_t)d[F_A0 + 5];
    const bool stat = kLean || ci >= 0;
    uint32_t next = stat ? (uint32_t)ci : atomicAdd(claim, 1u);
    if (!stat) ++c.stat[3];
    for (;;) {
      if (aborted(c)) return false;
      const uint32_t i = next;
      uint32_t acc = 0;
      int b = 0, n = 0, s = 0;
      for (; b < p.B; ++b) {
        s = __ldg(p.seq_lens + b);
        n = slices_of(p, s) * S::NKV;
        if (i < acc + (uint32_t)n) break;
        acc += (uint32_t)n;
      }
      if (b >= p.B) break;  // queue exhausted
      const int r = (int)(i - acc), per = n / S::NKV;
      const int g = r / per, j = r - g * per;
      if (j >= p.max_slots) {
        record_error(p, ERR_INDEX, c.sm, where_of(d), d[F_A0], (uint32_t)s, (uint32_t)p.max_ctx);
        c.hdr->abort = 1;
        return false;
      }
      const int t0 = j * p.split_len, t1 = min(s, t0 + p.split_len);
      if (!attn_item(d, l, b, g, t0, t1, j, d[F_A0 + 2] + g, d[F_A0 + 3], d[F_A0 + 1] + b * S::NKV + g))
        return false;
      if (stat) {
        next = i + n_cl;
      } else {
        if (c.wk >= 2u && !item_finished(c.wk - 2u)) return false;
        next = atomicAdd(claim, 1u);
        ++c.stat[3];
      }
    }
    return claim_end(d);
  }

  __device__ __forceinline__ bool claim_end(const int32_t* d) {
    int32_t it[32];
    for (int i = 0; i < 32; ++i) it[i] = d[i];
    it[F_OP] = W_CLAIM_END;
    it[F_WAIT0] = it[F_WAIT1] = -1;
    it[F_NSTAGE] = 0;
    return push(it);
  }

  // Claimer over the MoE tile queue ("Task scheduler": MOE_*_DRAIN claims the
  // next tile until the queue is empty).  mode 0: one queue of up/gate and down
  // tiles, each expert's down tiles one expert behind its up tiles --
  //   up(0) | up(1) down(0) | up(2) down(1) | ... | up(n-1) down(n-2) | down(n-1)
  // -- so a down tile rarely waits and no SM idles between the two phases;
  // every unit depends only on units with smaller indices, so the claimers
  // cannot deadlock.  mode 1: up/gate tiles only; mode 2: down tiles only.
  // Static assignment (default): claimer c of n takes units c, c + n, ...,
  // known as soon as the queue is, so the producer streams them back to back.
  // Otherwise claimer c takes unit c first without an atomic and later units
  // from the layer's claim counter, offset by n, each claim issued before the
  // current tile streams.
  // the layer whose routing this SM's MoE drains have already waited for,
  // and its active-expert count
  int routed_layer = -1, routed_n_act = 0;

  __device__ __forceinline__ bool moe_drain(const int32_t* d, int mode) {
    const int l = d[F_LAYER];
    constexpr MoePlan mp = gemv_plan_of<S, M>();  // (tile counts as plan_of)
    const int U = mp.up_tiles, DN = mp.dn_tiles;
    uint32_t* claim = p.bars + d[F_A0];
    const uint32_t n_claimers = (uint32_t)d[F_A0 + 5];
    const bool stat = kLean || d[F_A0 + 7] != 0;
    // the routing decides which expert rows to stream: wait for the queue
    // (once per layer: the down drain follows the up/gate drain's wait)
    int n_act;
    int4 first = make_int4(0, 0, 0, 0);
    int first_a = -1;
    if (routed_layer == l) {
      n_act = routed_n_act;
    } else {
      const int64_t t0 = p.stats ? gtimer() : 0;
      const bool ok = wait_counters(p, c, d[F_WAIT0], (uint32_t)d[F_TGT0], d[F_WAIT1], (uint32_t)d[F_TGT1], where_of(d));
      if (p.stats) c.stat[1] += gtimer() - t0;
      if (!ok) return false;
      // the active-expert count and a static claimer's first queue record in
      // one round trip (the record is read before knowing it is in range)
      if (stat && mode == 1 && (int)d[F_A0 + 4] / U < S::E) {
        first_a = (int)d[F_A0 + 4] / U;
        first = __ldcg(reinterpret_cast<const int4*>(p.act) + first_a);
      }
      n_act = min(__ldcg(p.qlen), S::E);
      routed_layer = l;
      routed_n_act = n_act;
    }
    const uint32_t total = (uint32_t)n_act * (mode == 0 ? U + DN : mode == 1 ? U : DN);
    uint32_t cur = (uint32_t)d[F_A0 + 4];
    // static assignment: units cur, cur + n, ...; the down units start after
    // the last up unit, so the claimers with an extra up/gate tile get no
    // extra down tile
    if (d[F_A0 + 7] == 1 && mode == 2)
      cur = (cur + n_claimers - ((uint32_t)n_act * U) % n_claimers) % n_claimers;
    uint32_t nxt = 0;
    if (cur < total) {
      if (stat) {
        nxt = cur + n_claimers;
      } else {
        nxt = n_claimers + atomicAdd(claim, 1u);
        ++c.stat[3];
      }
    }
    bool carried = false;  // the last unit carried the drain's signal
    int cached_a = first_a, dn_a = -1;
    int4 info = first;
    int32_t dn_slot[kTB] = {}, dn_wt[kTB] = {};  // a down tile's rows: output slot and routing weight
    while (cur < total) {
      if (aborted(c)) return false;
      bool up;
      int a, t;
      if (mode == 1) {
        up = true; a = (int)cur / U; t = (int)cur - a * U;
      } else if (mode == 2) {
        up = false; a = (int)cur / DN; t = (int)cur - a * DN;
      } else if ((int)cur < U) {
        up = true; a = 0; t = (int)cur;
      } else {
        const int j = (int)cur - U, blk = j / (U + DN), r = j - blk * (U + DN);
        if (blk < n_act - 1) {
          up = r < U;
          a = up ? blk + 1 : blk;
          t = up ? r : r - U;
        } else {
          up = false; a = n_act - 1; t = r;
        }
      }
      if (a != cached_a) {  // {expert, first row, rows} of active expert a
        info = __ldcg(reinterpret_cast<const int4*>(p.act) + a);
        cached_a = a;
      }
      const int e = info.x, row0 = info.y, nrows = info.z;
      if (e < 0 || e >= S::E || row0 < 0 || nrows < 1 || row0 + nrows > p.B * S::K) {
        record_error(p, ERR_INDEX, c.sm, where_of(d), d[F_A0], (uint32_t)cur, total);
        c.hdr->abort = 1;
        return false;
      }
      int32_t it[32];
      for (int k = 0; k < 32; ++k) it[k] = d[k];
      it[F_A0] = e;
      it[F_A0 + 1] = t;
      it[F_A0 + 2] = row0;
      it[F_A0 + 3] = nrows;
      it[F_WAIT1] = -1;
      it[F_SIG1] = -1;
      if (up) {
        it[F_OP] = W_UP_TILE;
        it[F_WAIT0] = d[F_A0 + 2];  // explicit gather barrier (or -1)
        it[F_TGT0] = d[F_A0 + 3];
        it[F_SIG0] = d[F_A0 + 1] + e;
        it[F_NSTAGE] = mp.up_stages * gemv_passes(nrows);
      } else {
        it[F_OP] = W_DOWN_TILE;
        it[F_WAIT0] = d[F_A0 + 1] + e;  // every up tile of expert e
        it[F_TGT0] = U;
        it[F_SIG0] = -1;
        it[F_NSTAGE] = mp.dn_stages * gemv_passes(nrows);
        // at most kTB rows: each row's (row b, choice j) slot and weight travel
        // with the item, so the epilogue waits on no load
        if (nrows <= kTB) {
          if (a != dn_a) {
#pragma unroll
            for (int t = 0; t < kTB; ++t) {
              int ds = t < nrows ? __ldcg(p.perm + row0 + t) : 0;
              if (ds < 0 || ds >= p.B * S::K) ds = 0;  // only after a failed step
              dn_slot[t] = ds;
            }
#pragma unroll
            for (int t = 0; t < kTB; ++t)
              dn_wt[t] = t < nrows ? __float_as_int(__ldcg(p.topk_w + (int64_t)l * p.MB * S::K + dn_slot[t])) : 0;
            dn_a = a;
          }
#pragma unroll
          for (int t = 0; t < kTB; ++t) {
            it[F_A0 + 8 + t] = dn_slot[t];
            it[F_A0 + 10 + t] = dn_wt[t];
          }
        }
      }
      // A static claimer's last unit carries the drain's own completion
      // signal (the storer publishes it after the tile): no claim-end item.
      if (stat && nxt >= total) {
        if (!up) {
          it[F_SIG0] = d[F_SIG0];
          it[F_SIG1] = d[F_SIG1];
          carried = true;
        } else if (d[F_SIG1] < 0) {
          it[F_SIG1] = d[F_SIG0];
          carried = true;
        }
      }
      if (mode_tc(M) && nrows > kTB) {
        // one item of nkb k-blocks: the expert's gate/up or down rows against
        // its routed rows (their hi/lo rows start at row 2 row0; FP8 experts:
        // their E4M3 term rows at row kTcF8Terms row0)
        constexpr bool f8 = M == kModeTcFp8;
        constexpr int kk = f8 ? kTcK8 : kTcK, nt = f8 ? kTcF8Terms : 2;
        const int nb = f8 ? p.tc_nb8 : p.tc_nb;
        const int64_t le = (int64_t)l * S::E + e;
        constexpr uint32_t ab = kTcMoeRows * kTcK * 2;  // 128 rows of 128 bytes (BF16 or FP8)
        const int nkb = up ? S::H / kk : S::I / kk, kps = tc_kblocks_per_stage(ab, nb);
        it[F_NSTAGE] = (nkb + kps - 1) / kps;
        it[F_A0 + 13] = nkb;
        if (!push(it)) return false;
        if (up) {
          if (!tc_stages(it, nullptr, 0, (int)(le * S::I + t * mp.up_tile), true, f8 ? &p.tm_xg8 : &p.tm_xgb, 0,
                         nt * row0, nkb, ab, kk, nb))
            return false;
        } else if (!tc_stages(it, &p.tm_wd, 0, (int)(le * S::H + t * mp.dn_tile), false, f8 ? &p.tm_u8 : &p.tm_ub, 0,
                              nt * row0, nkb, ab, kk, nb)) {
          return false;
        }
      } else {
        if (!push(it)) return false;
        for (int ps = gemv_passes(nrows); ps > 0; --ps)
          if (!tile_stages(l, e, t, up)) return false;
      }
      cur = nxt;
      if (cur < total) {
        if (stat) {
          nxt = cur + n_claimers;
        } else {
          nxt = n_claimers + atomicAdd(claim, 1u);
          ++c.stat[3];
        }
      }
    }
    return carried || claim_end(d);
  }

  // The weight stages of tile t of expert e: up/gate stages of up_half gate
  // rows and as many up rows, or down stages of dn_rows rows of W_down[e].
  // FP8 rows are 1 byte per weight: a row of K weights is K / 2 16-bit units.
  // FP4 stages: 16 rows (up/gate: 8 gate, then 8 up) of K/2 bytes of E2M1
  // codes, then the same rows' K/16 block scales; their row scales go to the
  // slot's scale area.  All on the stage's one full barrier.
  __device__ __forceinline__ bool tile_stages4(int l, int e, int t, bool up) {
    constexpr int R = kFp4StageRows;
    constexpr MoePlan mp = S::mp4;
    const int64_t le = (int64_t)l * S::E + e;
    const uint8_t* wg = reinterpret_cast<const uint8_t*>(p.wg);
    const uint8_t* wu = reinterpret_cast<const uint8_t*>(p.wu);
    const uint8_t* wd = reinterpret_cast<const uint8_t*>(p.wd);
    const int nst = up ? mp.up_stages : mp.dn_stages;
    for (int s = 0; s < nst; ++s) {
      int slot;
      if (!acquire_stage(slot)) return false;
      uint64_t* fb = &c.hdr->full[slot];
      uint8_t* dst = stage(slot);
      if (up) {
        constexpr uint32_t cb = (R / 2) * S::H / 2, bb = (R / 2) * S::H / 16, sb = (R / 2) * 4;
        const int64_t r0 = le * S::I + t * mp.up_tile + s * (R / 2);  // row of [L][E][I]
        mbar_expect_tx(fb, 2 * (cb + bb + sb));
        bulk_g2s_hint(dst, wg + r0 * (S::H / 2), cb, fb, stream_policy);
        bulk_g2s_hint(dst + cb, wu + r0 * (S::H / 2), cb, fb, stream_policy);
        bulk_g2s_hint(dst + 2 * cb, p.bg + r0 * (S::H / 16), bb, fb, stream_policy);
        bulk_g2s_hint(dst + 2 * cb + bb, p.bu + r0 * (S::H / 16), bb, fb, stream_policy);
        bulk_g2s(c.hdr->scl[slot], p.sg + r0, sb, fb);
        bulk_g2s(c.hdr->scl[slot] + R / 2, p.su + r0, sb, fb);
      } else {  // dn_rows rows: whole 16-row groups
        constexpr uint32_t cb = mp.dn_rows * S::I / 2, bb = mp.dn_rows * S::I / 16, sb = mp.dn_rows * 4;
        const int64_t r0 = le * S::H + t * mp.dn_tile + s * mp.dn_rows;  // row of [L][E][H]
        mbar_expect_tx(fb, cb + bb + sb);
        bulk_g2s_hint(dst, wd + r0 * (S::I / 2), cb, fb, stream_policy);
        bulk_g2s_hint(dst + cb, p.bd + r0 * (S::I / 16), bb, fb, stream_policy);
        bulk_g2s(c.hdr->scl[slot], p.sd + r0, sb, fb);
      }
      ++c.st;
    }
    return true;
  }

  __device__ __forceinline__ bool tile_stages(int l, int e, int t, bool up) {
    if constexpr (mode_fp4(M)) return tile_stages4(l, e, t, up);
    constexpr bool fp8 = mode_fp8(M) || M == kModeTcFp8;
    constexpr MoePlan mp = gemv_plan_of<S, M>();
    const int64_t le = (int64_t)l * S::E + e;
    constexpr int eb = fp8 ? 1 : 2;  // bytes per weight
    if (!up && !fp8) {
      const uint16_t* base = reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(p.wd) +
                                                               le * S::H * S::I * eb);
      return load_rows(base, S::I, S::I, t * mp.dn_tile, mp.dn_tile, mp.dn_rows);
    }
    if (!up) {
      // FP8 down stages: dn_rows rows of I bytes and their dn_rows scales
      const uint8_t* wd = reinterpret_cast<const uint8_t*>(p.wd) + le * S::H * S::I;
      for (int s = 0; s < mp.dn_stages; ++s) {
        int slot;
        if (!acquire_stage(slot)) return false;
        uint64_t* fb = &c.hdr->full[slot];
        const int r0 = t * mp.dn_tile + s * mp.dn_rows;
        const uint32_t bytes = (uint32_t)mp.dn_rows * S::I;
        mbar_expect_tx(fb, bytes + (uint32_t)mp.dn_rows * 4);
        bulk_g2s_hint(stage(slot), wd + (int64_t)r0 * S::I, bytes, fb, stream_policy);
        bulk_g2s(c.hdr->scl[slot], p.sd + le * S::H + r0, (uint32_t)mp.dn_rows * 4, fb);
        ++c.st;
      }
      return true;
    }
    const uint8_t* wg = reinterpret_cast<const uint8_t*>(p.wg);
    const uint8_t* wu = reinterpret_cast<const uint8_t*>(p.wu);
    for (int s = 0; s < mp.up_stages; ++s) {
      int slot;
      if (!acquire_stage(slot)) return false;
      uint64_t* fb = &c.hdr->full[slot];
      uint8_t* dst = stage(slot);
      const int r0 = t * mp.up_tile + s * mp.up_half;
      const uint32_t half = (uint32_t)mp.up_half * S::H * eb;
      const uint32_t sb = fp8 ? (uint32_t)mp.up_half * 4 : 0u;  // FP8: scales
      mbar_expect_tx(fb, 2 * half + 2 * sb);
      bulk_g2s_hint(dst, wg + (le * S::I + r0) * S::H * eb, half, fb, stream_policy);
      bulk_g2s_hint(dst + half, wu + (le * S::I + r0) * S::H * eb, half, fb, stream_policy);
      if (sb) {
        bulk_g2s(c.hdr->scl[slot], p.sg + le * S::I + r0, sb, fb);
        bulk_g2s(c.hdr->scl[slot] + mp.up_half, p.su + le * S::I + r0, sb, fb);
      }
      ++c.st;
    }
    return true;
  }

  // A dense FFN tile ("Tasks": FFN_UPGATE_ACT, FFN_DOWN): a static task for
  // tile A0 of the layer's one FFN (stored as expert 0), over every row of
  // the batch; the same work item as an MoE tile, with each row its own slot
  // and weight 1 (the dense flag A12).
  __device__ __forceinline__ bool ffn_tile(const int32_t* d) {
    constexpr MoePlan mp = plan_of<S, M>();
    const bool up = d[F_OP] == OP_FFN_UPGATE_ACT;
    int32_t it[32];
    for (int k = 0; k < 32; ++k) it[k] = d[k];
    it[F_OP] = up ? W_UP_TILE : W_DOWN_TILE;
    it[F_A0] = 0;          // expert
    it[F_A0 + 1] = d[F_A0];  // tile
    it[F_A0 + 2] = 0;      // first row
    it[F_A0 + 3] = p.B;    // rows
    it[F_A0 + 12] = 1;     // dense
    for (int t = 0; t < kTB; ++t) {
      it[F_A0 + 8 + t] = t;  // row b's output goes to slot b (one choice per row)
      it[F_A0 + 10 + t] = __float_as_int(1.f);
    }
    it[F_NSTAGE] = (up ? mp.up_stages : mp.dn_stages) * gemv_passes(p.B);
    if (!push(it)) return false;
    for (int ps = gemv_passes(p.B); ps > 0; --ps)
      if (!tile_stages(d[F_LAYER], 0, d[F_A0], up)) return false;
    return true;
  }

  __device__ __forceinline__ bool passthrough(const int32_t* d) {
    int32_t it[32];
    for (int i = 0; i < 32; ++i) it[i] = d[i];
    it[F_NSTAGE] = 0;
    return push(it);
  }

  __device__ __forceinline__ void run() {
    if ((threadIdx.x & 31) != 0) return;
    stream_policy = l2_evict_first_policy();
    const int n = p.sched[2 * c.sm + 1];
    Hdr* H = c.hdr;
    bool ok = true;
    for (int i = 0; i < n && ok; ++i) {
      const int slot = i % kDescRing;
      if (!mbar_wait(p, c, &H->dfull[slot], (i / kDescRing) & 1)) {
        ok = false;
        break;
      }
      // the controller's next TMA copy overwrites this slot: explicit
      // shared-memory loads, then a cross-proxy fence, then the release
      int32_t d[32];
      const uint32_t da = smem_u32(H->desc[slot]);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint4 v = lds128(da + 16u * k);
        d[4 * k] = (int32_t)v.x; d[4 * k + 1] = (int32_t)v.y; d[4 * k + 2] = (int32_t)v.z; d[4 * k + 3] = (int32_t)v.w;
      }
      fence_proxy_async_smem();
      mbar_arrive(&H->dempty[slot]);
      p.prog[c.sm * 8 + 3] = (uint32_t)(i + 1);
      if (d[F_POS] != i) {
        record_error(p, ERR_RING, c.sm, where_of(d), i, (uint32_t)d[F_POS], (uint32_t)n);
        H->abort = 1;
        ok = false;
        break;
      }
      switch (d[F_OP]) {
        case OP_QKV_PROJ:
        case OP_O_PROJ:
        case OP_ROUTER_GEMM:
        case OP_LM_HEAD: ok = dense(d); break;
        case OP_ATTN_DECODE: ok = attn_decode(d); break;
        case OP_ATTN_DRAIN: ok = attn_drain(d); break;
        case OP_MOE_UPGATE_ACT_DRAIN: ok = moe_drain(d, kLean ? 1 : d[F_A0 + 6]); break;
        case OP_MOE_DOWN_DRAIN: ok = moe_drain(d, 2); break;
        case OP_FFN_UPGATE_ACT:
        case OP_FFN_DOWN: ok = ffn_tile(d); break;
        default: ok = passthrough(d); break;
      }
    }
    if (ok) {
      int32_t ex[32];
      for (int k = 0; k < 32; ++k) ex[k] = 0;
      ex[F_OP] = W_EXIT;
      ex[F_WAIT0] = ex[F_WAIT1] = ex[F_SIG0] = ex[F_SIG1] = -1;
      push(ex);
      if (p.stats)
        for (int k = 0; k < 4; ++k) p.stats[(int64_t)c.sm * kStats + 4 + k] = c.stat[k];
      return;
    }
    // aborting: wait (bounded) for the copies already issued into the stage ring
    const uint32_t first = c.st > (uint32_t)kStages ? c.st - kStages : 0;
    for (uint32_t s = first; s < c.st; ++s) {
      const int64_t t0 = gtimer();
      while (!mbar_try_wait(&H->full[s % kStages], (s / kStages) & 1) && gtimer() - t0 < p.watchdog_ns) {
      }
    }
  }
};

// ======================================================================
// consumers
// ======================================================================
template <class S, int M>
struct Consumer {
  // the lean builds leave out the tasks of unfused schedules
  static constexpr bool kLean = mode_lean(M);
  const Params& p;
  Ctx c;
  Scratch<S>& sm;
  int ct, cw, lane;
  uint32_t tmem = 0;       // kModeTc: TMEM address of the accumulator
  uint32_t acc_phase = 0;  // kModeTc: parity of the accumulator's next completion

  // --- the stage ring
  __device__ __forceinline__ bool stage_wait(int& slot) {
    slot = c.st % kStages;
    const int64_t t0 = (p.stats && ct == 0) ? gtimer() : 0;
    const bool ok = mbar_wait(p, c, &c.hdr->full[slot], (c.st / kStages) & 1);
    if (p.stats && ct == 0) c.stat[1] += gtimer() - t0;
    return ok;
  }
  // The stage goes back to the producer, whose next TMA copy overwrites it.
  // Every read of a stage is an explicit shared-memory load (ld.shared,
  // ldmatrix), which the release orders before the arrival.
  __device__ __forceinline__ void stage_release(int slot) {
    if constexpr (mode_tc(M)) {  // the stage's two arrivals, after every consumer warp's reads
      consumers_sync();
      if (ct == 0) mbar_arrive_n(&c.hdr->empty[slot], 2);
    } else {
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.hdr->empty[slot]);
    }
    ++c.st;
  }
  __device__ __forceinline__ const uint8_t* stage(int slot) const { return c.stages + (size_t)slot * kStageBytes; }

  // ---------------------------------------------------------- GEMV core
  // out[t][r] = W[r][:] . xs[t][:] for the rows of one stage (warp per row).
  // xs row t holds the activation as [half][chunk][4]: lane c reads the two
  // halves of its 8-element chunk with two conflict-free 16-byte loads.
  template <int K>
  __device__ __forceinline__ void gemv_rows(const uint16_t* W, int rows, int tb, float* out) {
    constexpr int C = K / 8;
    constexpr int CPL = (C + 31) / 32;
    const float4* xs4 = reinterpret_cast<const float4*>(sm.xs);
    for (int r = cw; r < rows; r += kConsumerWarps) {
      float acc0[kTB], acc1[kTB];
#pragma unroll
      for (int t = 0; t < kTB; ++t) acc0[t] = acc1[t] = 0.f;
      const uint32_t wr = smem_u32(W + (size_t)r * K);
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        const int cc = lane + 32 * j;
        if (C % 32 == 0 || cc < C) {
          const uint4 w = lds128(wr + 16u * cc);
#pragma unroll
          for (int t = 0; t < kTB; ++t)
            if (t < tb) {
              const float4 a = xs4[t * 2 * C + cc], b = xs4[t * 2 * C + C + cc];
              acc0[t] = fmaf(bf16_lo(w.x), a.x, acc0[t]);
              acc1[t] = fmaf(bf16_hi(w.x), a.y, acc1[t]);
              acc0[t] = fmaf(bf16_lo(w.y), a.z, acc0[t]);
              acc1[t] = fmaf(bf16_hi(w.y), a.w, acc1[t]);
              acc0[t] = fmaf(bf16_lo(w.z), b.x, acc0[t]);
              acc1[t] = fmaf(bf16_hi(w.z), b.y, acc1[t]);
              acc0[t] = fmaf(bf16_lo(w.w), b.z, acc0[t]);
              acc1[t] = fmaf(bf16_hi(w.w), b.w, acc1[t]);
            }
        }
      }
#pragma unroll
      for (int t = 0; t < kTB; ++t)
        if (t < tb) acc0[t] = warp_sum(acc0[t] + acc1[t]);
      if (lane == 0)
#pragma unroll
        for (int t = 0; t < kTB; ++t)
          if (t < tb) out[t * kMaxStageRows + r] = acc0[t];
    }
  }

  // activation rows [kTB*chunk, kTB*chunk + tb) of the item into sm.xs (fp32)
  template <int K>
  __device__ __forceinline__ void load_x(int op, const int32_t* w, int chunk, int tb) {
    static_assert(K <= xs_row<S>(), "kTB activation rows of K fit the cache");
    constexpr int C = K / 4;  // float4 per row
    float4* xs4 = reinterpret_cast<float4*>(sm.xs);
    for (int i = ct; i < tb * C; i += kConsumerThreads) {
      const int t = i / C, cc = i - t * C;
      const float* src = x_src(op, w, kTB * chunk + t);
      // source float4 cc = elements [4cc, 4cc+4): chunk cc/2, half cc%2
      xs4[t * C + (cc & 1) * (C / 2) + (cc >> 1)] = __ldcg(reinterpret_cast<const float4*>(src) + cc);
    }
  }

  // the activation row `tok` of an item's input
  __device__ __forceinline__ const float* x_src(int op, const int32_t* w, int tok) {
    switch (op) {
      case OP_O_PROJ:
        return p.attn_out + (int64_t)tok * S::NQ * S::D + (int64_t)w[F_A0 + 2] * S::G * S::D;
      case W_UP_TILE: {
        const int row = w[F_A0 + 2] + tok;
        if (w[F_A0 + 12]) return p.x + (int64_t)row * S::H;  // dense: the rows are the batch
        // (the tensor-core builds' gather writes only the tcgen05 operand rows)
        if (!mode_tc(M) && p.explicit_gather) return p.xg + (int64_t)row * S::H;
        const int pr = __ldcg(p.perm + row);
        int b = pr / S::K;
        if (pr < 0 || b >= p.B) b = 0;  // only after a failed step
        return p.x + (int64_t)b * S::H;
      }
      case W_DOWN_TILE:
        return p.u + (int64_t)(w[F_A0 + 2] + tok) * S::I;
      default:
        return p.x + (int64_t)tok * S::H;
    }
  }

  // The activation rows an item reads, as a tag: xs is reloaded only when
  // the tag changes (consecutive items of one layer share their input).
  __device__ __forceinline__ void x_tag(int op, const int32_t* w, int chunk, int32_t (&tag)[4]) {
    const int l = w[F_LAYER];
    switch (op) {
      case OP_O_PROJ: tag[0] = 2; tag[1] = w[F_A0 + 2]; tag[2] = kTB * chunk; tag[3] = l; break;
      case W_UP_TILE:
        if (p.B == 1) {  // one row: the layer input itself, as for QKV and the router
          tag[0] = 1; tag[1] = 0; tag[2] = 0; tag[3] = l;
        } else {
          tag[0] = 3; tag[1] = w[F_A0 + 2] + kTB * chunk; tag[2] = w[F_A0 + 3]; tag[3] = l;
        }
        break;
      case W_DOWN_TILE: tag[0] = 4; tag[1] = w[F_A0 + 2] + kTB * chunk; tag[2] = w[F_A0 + 3]; tag[3] = l; break;
      default: tag[0] = 1; tag[1] = kTB * chunk; tag[2] = l == p.L ? 1 : 0; tag[3] = l; break;
    }
  }

  // epilogue of one stage: rows [r_first, r_first + rows) of the item's output,
  // activation rows [4*chunk, 4*chunk + tb)
  __device__ __forceinline__ void epilogue(int op, const int32_t* w, int s, int rows, int chunk, int tb, const float* out) {
    const int l = w[F_LAYER];
    switch (op) {
      case OP_QKV_PROJ: {
        // RoPE in the epilogue, then the new K/V into the pool ("Tasks":
        // QKV_PROJ applies RoPE in-register before writing back)
        const int half = rows / 2;
        for (int i = ct; i < tb * half; i += kConsumerThreads) {
          const int t = i / half, r = 2 * (i - t * half);
          const int row = w[F_A0] + s * S::SR_H + r;
          const int b = kTB * chunk + t;
          float v0 = out[t * kMaxStageRows + r], v1 = out[t * kMaxStageRows + r + 1];
          const int head = row / S::D, dd = row - head * S::D;
          const int pos = __ldg(p.seq_lens + b) - 1;
          if (head < S::NQ + S::NKV) {  // rotate q and k: pair (dd, dd+1) by pos * base^(-dd/D)
            // the angle is reduced modulo 2 pi in double, then sin/cos in float
            const double ang = (double)pos * sm.rope_theta[dd / 2];
            const double red = ang - 6.283185307179586 * rint(ang * 0.15915494309189535);
            float s0, c0;
            sincosf((float)red, &s0, &c0);
            const float r0 = v0 * c0 - v1 * s0, r1 = v0 * s0 + v1 * c0;
            v0 = r0;
            v1 = r1;
          }
          if (head < S::NQ) {
            float* qd = p.q + ((int64_t)b * S::NQ + head) * S::D + dd;
            qd[0] = v0;
            qd[1] = v1;
          } else if (pos >= 0) {
            const bool is_v = head >= S::NQ + S::NKV;
            const int g = head - S::NQ - (is_v ? S::NKV : 0);
            const uint32_t packed = (uint32_t)f_bf16(v0) | ((uint32_t)f_bf16(v1) << 16);
            *reinterpret_cast<uint32_t*>(p.kvnew + (((int64_t)b * 2 + (is_v ? 1 : 0)) * S::NKV + g) * S::D + dd) = packed;
            const int lp = pos / S::P;
            int page = lp < p.max_pages ? __ldg(p.block_tables + (int64_t)b * p.max_pages + lp) : -1;
            if (page < 0 || page >= p.num_pages) {
              record_error(p, ERR_PAGE, c.sm, where_of(w), lp, (uint32_t)page, (uint32_t)p.num_pages);
            } else {
              uint16_t* pool = is_v ? p.vpool : p.kpool;
              const int64_t o = ((((int64_t)l * p.num_pages + page) * S::NKV + g) * S::P + pos % S::P) * S::D + dd;
              *reinterpret_cast<uint32_t*>(pool + o) = packed;
            }
          }
        }
        break;
      }
      case OP_ROUTER_GEMM:
        for (int i = ct; i < tb * rows; i += kConsumerThreads) {
          const int t = i / rows, r = i - t * rows;
          const int e = w[F_A0] + s * S::SR_H + r, b = kTB * chunk + t;
          p.rlog[((int64_t)l * p.MB + b) * S::E + e] = out[t * kMaxStageRows + r] + (p.rbias ? p.rbias[e] : 0.f);
        }
        break;
      case OP_LM_HEAD:
        for (int i = ct; i < tb * rows; i += kConsumerThreads) {
          const int t = i / rows, r = i - t * rows;
          const int v = w[F_A0] + s * S::SR_H + r, b = kTB * chunk + t;
          p.logits[(int64_t)b * p.V + v] = out[t * kMaxStageRows + r];
        }
        break;
      case OP_O_PROJ:
        for (int i = ct; i < tb * rows; i += kConsumerThreads) {
          const int t = i / rows, r = i - t * rows;
          const int n = w[F_A0] + s * S::SR_O + r, b = kTB * chunk + t;
          p.opart[(((int64_t)(l & 1) * S::NKV + w[F_A0 + 2]) * p.MB + b) * S::H + n] = out[t * kMaxStageRows + r];
        }
        break;
      case W_UP_TILE: {
        // SiLU(gate) * up in the epilogue ("Tasks": the SiLU-and-multiply)
        constexpr int hu = S::mp.up_half;
        for (int i = ct; i < tb * hu; i += kConsumerThreads) {
          const int t = i / hu, r = i - t * hu;
          const float gte = out[t * kMaxStageRows + r], upv = out[t * kMaxStageRows + hu + r];
          const float act = gte / (1.f + expf(-gte)) * upv;
          const int row = w[F_A0 + 2] + kTB * chunk + t;
          const int col = w[F_A0 + 1] * S::mp.up_tile + s * hu + r;
          p.u[(int64_t)row * S::I + col] = act;
        }
        break;
      }
      case W_DOWN_TILE:
        // the output goes to the (row b, slot j) it belongs to, times its router weight
        for (int i = ct; i < tb * rows; i += kConsumerThreads) {
          const int t = i / rows, r = i - t * rows;
          const int row = w[F_A0 + 2] + kTB * chunk + t;
          const bool dense = w[F_A0 + 12] != 0;  // row b is slot b, weight 1
          int slot = dense ? row : __ldcg(p.perm + row);
          if (slot < 0 || slot >= p.B * S::K) slot = 0;  // only after a failed step
          const float wt = dense ? 1.f : __ldcg(p.topk_w + (int64_t)l * p.MB * S::K + slot);
          const int n = w[F_A0 + 1] * S::mp.dn_tile + s * S::mp.dn_rows + r;
          p.y[(int64_t)slot * S::H + n] = wt * out[t * kMaxStageRows + r];
        }
        break;
      default: break;
    }
  }

  // A GEMV item: stages of full weight rows, activation rows in passes of
  // kTB.  The producer streams the stages once per pass; each pass loads its
  // activation rows once and runs every stage against them.
  template <int K>
  __device__ __forceinline__ void gemv_item(const int32_t* w, int SR, int total_rows, int ntok) {
    const int op = w[F_OP];
    const int nchunk = (ntok + kTB - 1) / kTB;
    const int nst = w[F_NSTAGE] / nchunk;
    int buf = 0;
    for (int chunk = 0; chunk < nchunk; ++chunk) {
      const int tb = min(kTB, ntok - kTB * chunk);
      int32_t tag[4];
      x_tag(op, w, chunk, tag);
      if (!(tag[0] == sm.xtag[0] && tag[1] == sm.xtag[1] && tag[2] == sm.xtag[2] && tag[3] == sm.xtag[3])) {
        consumers_sync();  // every warp is done with the old rows
        if (!aborted(c)) load_x<K>(op, w, chunk, tb);
        consumers_sync();
        if (ct == 0) {
          sm.xtag[0] = tag[0]; sm.xtag[1] = tag[1]; sm.xtag[2] = tag[2]; sm.xtag[3] = tag[3];
        }
      }
      for (int s = 0; s < nst; ++s) {
        int slot;
        const bool ok = stage_wait(slot);
        const int rows = min(SR, total_rows - s * SR);
        const uint16_t* W = reinterpret_cast<const uint16_t*>(stage(slot));
        if (__all_sync(FULL, ok && !aborted(c))) gemv_rows<K>(W, rows, tb, sm.out[buf]);
        consumers_sync();
        if (!aborted(c)) epilogue(op, w, s, rows, chunk, tb, sm.out[buf]);
        buf ^= 1;
        stage_release(slot);
      }
    }
  }


  // Activation rows of an FP8 / FP4 expert tile as the B operand of f16 MMAs
  // (m16n8k16, the weights as A).  Column 2t of B is the f16 rounding of
  // activation row t, column 2t + 1 the f16 rounding of what that leaves
  // (x - hi): hi + lo carry about 22 bits of x, and the MMA accumulates in
  // fp32.  In one MMA, thread (n = lane / 4, q = lane % 4) holds the logical
  // k 2q, 2q+1, 2q+8, 2q+9; they stand for the physical elements
  // CH kc + (CH/4) q + 4 j + 0..3 of MMA j of CH-element chunk kc (CH = 64
  // for FP8, 128 for FP4): the elements one 16-byte load of a weight row
  // gives thread q.  Layout: uint4 [kc][j / 2][n][q] holding the (b0b1,
  // b2b3) words of MMAs 2(j/2) and 2(j/2) + 1.  An activation beyond the f16
  // range is reported as an error.
  template <int K, int CH>
  __device__ __forceinline__ void load_x_f16(int op, const int32_t* w, int tb) {
    static_assert(kTB <= 2 && K * 8 <= (int)sizeof(sm.xs), "the hi/lo columns of kTB rows of K fit the cache");
    constexpr int U = K / 8;  // 8-element units per row
    uint4* xb = reinterpret_cast<uint4*>(sm.xs);
    int bad = -1;
    for (int i = ct; i < tb * U; i += kConsumerThreads) {
      const int t = i / U, m = i - t * U;
      const float4* src = reinterpret_cast<const float4*>(x_src(op, w, t)) + 2 * m;
      const float4 a = __ldcg(src), b = __ldcg(src + 1);
      const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (fabsf(v[2 * k]) > 65504.f || fabsf(v[2 * k + 1]) > 65504.f) bad = 8 * m + 2 * k;
        hi[k] = f16x2_rn(v[2 * k], v[2 * k + 1]);
        const float2 h = f16x2_f32(hi[k]);
        lo[k] = f16x2_rn(v[2 * k] - h.x, v[2 * k + 1] - h.y);
      }
      constexpr int QS = CH / 4, JP = QS / 8;
      const int e = 8 * m, kc = e / CH, q = (e % CH) / QS, jp = (e % QS) / 8;
      const int at = (kc * JP + jp) * 16 + q;
      xb[at + 2 * t * 4] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      xb[at + (2 * t + 1) * 4] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    if (bad >= 0) record_error(p, ERR_RANGE, c.sm, where_of(w), bad, 0u, 65504u);
  }

  // FP8 expert tiles (batch <= kTB) on the tensor cores.  A stage's rows, 16
  // at a time, are the A operand of m16n8k16 MMAs (each E4M3 code converted
  // exactly to f16), the activations' hi/lo columns the B operand; the row
  // scale multiplies the finished fp32 dot product.  The same four teams of
  // two warps take the stages; a warp takes whole 16-row groups, or, when a
  // stage is one group, half of its chunks, the halves added through shared
  // memory.  A group pairs what one thread finishes: gate row i with up row
  // i (up/gate), rows 2i and 2i + 1 (down).
  static constexpr int kBarTeam0 = kBarConsumers + 1;  // named barriers of the teams' warp pairs
  template <int K, int TB>
  __device__ __forceinline__ void gemv_item_fp8(const int32_t* w, int SR, int ntok) {
    static_assert(K % 128 == 0, "FP8 rows in pairs of 64-byte chunks");
    static_assert(kTeamWarps == 2 && kTeams * 2 * kTB * 16 <= (int)(sizeof(sm.out) / sizeof(float)),
                  "partial sums of split stages fit the stage-output buffer");
    constexpr int NP = K / 128;  // pairs of 64-byte chunks per row
    const int op = w[F_OP];
    const int nst = w[F_NSTAGE];
    const int tb = ntok;
    const int g = lane >> 2, q = lane & 3;
    // epilogue inputs of activation row t = q, from the item
    int dslot = 0;
    float dwt = 0.f;
    if (op == W_DOWN_TILE && q < tb) {
      dslot = q == 0 ? w[F_A0 + 8] : w[F_A0 + 9];
      dwt = __int_as_float(q == 0 ? w[F_A0 + 10] : w[F_A0 + 11]);
    }
    int32_t tag[4];
    x_tag(op, w, 0, tag);
    tag[0] += 16;  // the same rows in the f16 hi/lo layout
    if (!(tag[0] == sm.xtag[0] && tag[1] == sm.xtag[1] && tag[2] == sm.xtag[2] && tag[3] == sm.xtag[3])) {
      if (!aborted(c)) load_x_f16<K, 64>(op, w, tb);
      consumers_sync();
      if (ct == 0) {
        sm.xtag[0] = tag[0]; sm.xtag[1] = tag[1]; sm.xtag[2] = tag[2]; sm.xtag[3] = tag[3];
      }
    }
    const int team = cw / kTeamWarps, tw = cw % kTeamWarps;
    const bool up = op == W_UP_TILE;
    const int ngroups = SR / 16;
    const bool split = ngroups < kTeamWarps;
    const bool bon = g < 2 * (TB == 1 ? 1 : tb);  // lanes that hold a B column
    const uint32_t xb_a = smem_u32(sm.xs) + (uint32_t)lane * 16u;
    float* red = &sm.out[0][0];  // [team][2][kTB][16]
    int it = 0;
    for (int s = team; s < nst; s += kTeams, ++it) {
      const uint32_t gs = c.st + (uint32_t)s;
      const int slot = gs % kStages;
      bool ok = s < kStages || mbar_wait(p, c, &c.hdr->empty[slot], ((gs / kStages) - 1) & 1);
      ok = __all_sync(FULL, ok && mbar_wait(p, c, &c.hdr->full[slot], (gs / kStages) & 1) && !aborted(c));
      const uint32_t st = smem_u32(stage(slot)) + (uint32_t)q * 16u;
      for (int grp = split ? 0 : tw; grp < ngroups; grp += split ? ngroups : kTeamWarps) {
        const int rlo = up ? 8 * grp + g : 16 * grp + 2 * g;
        const int rhi = up ? SR / 2 + 8 * grp + g : rlo + 1;
        const int m0 = split ? tw * NP / 2 : 0, m1 = split ? (tw + 1) * NP / 2 : NP;
        float d[4][4];  // one accumulator per MMA slot j: four independent chains
#pragma unroll
        for (int j = 0; j < 4; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.f;
        if (ok) {
          const uint32_t alo = st + (uint32_t)(rlo * K), ahi = st + (uint32_t)(rhi * K);
          for (int m = m0; m < m1; ++m) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int kc = 2 * m + h;
              const uint4 ul = lds128(alo + (uint32_t)(kc * 64)), uh = lds128(ahi + (uint32_t)(kc * 64));
              uint4 b01 = make_uint4(0u, 0u, 0u, 0u), b23 = b01;
              if (bon) {
                b01 = lds128(xb_a + (uint32_t)((2 * kc) * 256));
                b23 = lds128(xb_a + (uint32_t)((2 * kc + 1) * 256));
              }
              uint32_t a0, a1, a2, a3;
              e4m3x4_f16(ul.x, a0, a2);
              e4m3x4_f16(uh.x, a1, a3);
              mma_f16(d[0], a0, a1, a2, a3, b01.x, b01.y);
              e4m3x4_f16(ul.y, a0, a2);
              e4m3x4_f16(uh.y, a1, a3);
              mma_f16(d[1], a0, a1, a2, a3, b01.z, b01.w);
              e4m3x4_f16(ul.z, a0, a2);
              e4m3x4_f16(uh.z, a1, a3);
              mma_f16(d[2], a0, a1, a2, a3, b23.x, b23.y);
              e4m3x4_f16(ul.w, a0, a2);
              e4m3x4_f16(uh.w, a1, a3);
              mma_f16(d[3], a0, a1, a2, a3, b23.z, b23.w);
            }
          }
        }
        // column 2t + {0, 1} of rows g and g + 8: thread q = t holds both
        float vlo = (d[0][0] + d[1][0]) + (d[2][0] + d[3][0]) + ((d[0][1] + d[1][1]) + (d[2][1] + d[3][1]));
        float vhi = (d[0][2] + d[1][2]) + (d[2][2] + d[3][2]) + ((d[0][3] + d[1][3]) + (d[2][3] + d[3][3]));
        if (split) {
          float* rb = red + (team * 2 + (it & 1)) * kTB * 16;
          if (tw == 1 && q < tb) {
            rb[q * 16 + g] = vlo;
            rb[q * 16 + 8 + g] = vhi;
          }
          bar_sync(kBarTeam0 + team, 2 * 32);
          if (tw == 1) continue;
          if (q < tb) {
            vlo += rb[q * 16 + g];
            vhi += rb[q * 16 + 8 + g];
          }
        }
        if (ok && q < tb && !aborted(c)) {
          const float slo = c.hdr->scl[slot][rlo], shi = c.hdr->scl[slot][rhi];
          pair_epilogue(op, w, s, up ? 8 * grp + g : rlo, rhi, q, vlo * slo, vhi * shi, dslot, dwt);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_n(&c.hdr->empty[slot], kTeamArrivals);
    }
    c.st += (uint32_t)nst;
  }

  // FP4 expert tiles (batch <= kTB) on the tensor cores: each 16-row group
  // of a stage (one per up/gate stage, up to four per down stage) is one
  // group of m16n8k16 f16 MMAs.  A thread's 16-byte load of a row
  // holds 32 codes (two 16-input blocks) and feeds eight MMAs; each code pair
  // is converted exactly to f16 and multiplied (exactly: at most 6
  // significant bits, within the f16 range) by its block's E4M3 scale before
  // the MMA.  The two warps of a team take half of the stage's 128-input
  // chunks each and add their sums through shared memory; the row scale
  // multiplies the finished dot product.
  template <int K, int TB>
  __device__ __forceinline__ void gemv_item_fp4(const int32_t* w, int ntok) {
    static_assert(K % 128 == 0, "FP4 rows in 128-input chunks");
    static_assert(kTeamWarps == 2 && kTeams * 2 * kTB * 16 <= (int)(sizeof(sm.out) / sizeof(float)),
                  "partial sums of the stages fit the stage-output buffer");
    constexpr int R = kFp4StageRows, NKC = K / 128;  // rows of a group, 128-input chunks of a row
    const int op = w[F_OP];
    const int nst = w[F_NSTAGE];
    const int tb = ntok;
    const int g = lane >> 2, q = lane & 3;
    int dslot = 0;
    float dwt = 0.f;
    if (op == W_DOWN_TILE && q < tb) {
      dslot = q == 0 ? w[F_A0 + 8] : w[F_A0 + 9];
      dwt = __int_as_float(q == 0 ? w[F_A0 + 10] : w[F_A0 + 11]);
    }
    int32_t tag[4];
    x_tag(op, w, 0, tag);
    tag[0] += 32;  // the same rows in the FP4 hi/lo layout
    if (!(tag[0] == sm.xtag[0] && tag[1] == sm.xtag[1] && tag[2] == sm.xtag[2] && tag[3] == sm.xtag[3])) {
      if (!aborted(c)) load_x_f16<K, 128>(op, w, tb);
      consumers_sync();
      if (ct == 0) {
        sm.xtag[0] = tag[0]; sm.xtag[1] = tag[1]; sm.xtag[2] = tag[2]; sm.xtag[3] = tag[3];
      }
    }
    const int team = cw / kTeamWarps, tw = cw % kTeamWarps;
    const bool up = op == W_UP_TILE;
    // a down stage holds ng 16-row groups (codes of all its rows, then their
    // block scales): with kFp4DownGroups of them every team takes one group of
    // every stage (and each warp stands for one arrival), else the teams take
    // stages in turn
    constexpr MoePlan mp4 = S::mp4;
    static_assert(kFp4DownGroups == kTeams, "one group of a down stage per team");
    const int rows = up ? R : mp4.dn_rows, ng = rows / R, cbytes = rows * K / 2;
    const bool spread = ng == kTeams;
    const int s0 = spread ? 0 : team, ds = spread ? 1 : kTeams, g0 = spread ? team : 0, dg = spread ? kTeams : 1;
    const int arrivals = spread ? kConsumerWarps / (kTeams * kTeamWarps) : kTeamArrivals;
    const int c0 = tw * NKC / 2, c1 = (tw + 1) * NKC / 2;
    const bool bon = g < 2 * (TB == 1 ? 1 : tb);
    const uint32_t xb_a = smem_u32(sm.xs) + (uint32_t)lane * 16u;
    float* red = &sm.out[0][0];  // [team][2][kTB][16]
    int it = 0;
    for (int s = s0; s < nst; s += ds) {
      const uint32_t gs = c.st + (uint32_t)s;
      const int slot = gs % kStages;
      bool ok = s < kStages || mbar_wait(p, c, &c.hdr->empty[slot], ((gs / kStages) - 1) & 1);
      ok = __all_sync(FULL, ok && mbar_wait(p, c, &c.hdr->full[slot], (gs / kStages) & 1) && !aborted(c));
      const uint32_t st = smem_u32(stage(slot));
      for (int gi = g0; gi < ng; gi += dg, ++it) {
        // gate/up row g and up row g (rows g, R/2 + g), or rows 2g, 2g + 1 of group gi
        const int rlo = up ? g : R * gi + 2 * g, rhi = up ? R / 2 + g : rlo + 1;
        float d[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.f;
        if (ok) {
          const uint32_t alo = st + (uint32_t)(rlo * (K / 2) + q * 16), ahi = st + (uint32_t)(rhi * (K / 2) + q * 16);
          const uint32_t blo = st + (uint32_t)(cbytes + rlo * (K / 16) + q * 2);
          const uint32_t bhi = st + (uint32_t)(cbytes + rhi * (K / 16) + q * 2);
          for (int kc = c0; kc < c1; ++kc) {
            const uint4 ul = lds128(alo + (uint32_t)(kc * 64)), uh = lds128(ahi + (uint32_t)(kc * 64));
            // the scales of blocks 2q (MMAs 0-3) and 2q + 1 (MMAs 4-7) of the chunk
            uint32_t sl, sh, unused;
            e4m3x4_f16(lds_u16(blo + (uint32_t)(kc * 8)), sl, unused);
            e4m3x4_f16(lds_u16(bhi + (uint32_t)(kc * 8)), sh, unused);
            const uint32_t sl0 = half_bcast(sl, 0x1010u), sl1 = half_bcast(sl, 0x3232u);
            const uint32_t sh0 = half_bcast(sh, 0x1010u), sh1 = half_bcast(sh, 0x3232u);
            uint4 b[4];
#pragma unroll
            for (int jp = 0; jp < 4; ++jp)
              b[jp] = bon ? lds128(xb_a + (uint32_t)((kc * 4 + jp) * 256)) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t wl[4] = {ul.x, ul.y, ul.z, ul.w}, wh[4] = {uh.x, uh.y, uh.z, uh.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              // MMA j: codes 4j .. 4j+3 of the thread's 32 (bytes 2j, 2j+1)
              const uint32_t cl = (j & 1) ? wl[j >> 1] >> 16 : wl[j >> 1];
              const uint32_t chh = (j & 1) ? wh[j >> 1] >> 16 : wh[j >> 1];
              uint32_t a0, a1, a2, a3;
              e2m1x4_f16(cl, a0, a2);
              e2m1x4_f16(chh, a1, a3);
              const uint32_t fl = j < 4 ? sl0 : sl1, fh = j < 4 ? sh0 : sh1;
              a0 = hmul2(a0, fl);
              a2 = hmul2(a2, fl);
              a1 = hmul2(a1, fh);
              a3 = hmul2(a3, fh);
              const uint32_t b0 = (j & 1) ? b[j >> 1].z : b[j >> 1].x, b1 = (j & 1) ? b[j >> 1].w : b[j >> 1].y;
              mma_f16(d[j & 3], a0, a1, a2, a3, b0, b1);
            }
          }
        }
        // columns 2t + {0, 1} of rows g and g + 8: thread q = t holds both
        float vlo = (d[0][0] + d[1][0]) + (d[2][0] + d[3][0]) + ((d[0][1] + d[1][1]) + (d[2][1] + d[3][1]));
        float vhi = (d[0][2] + d[1][2]) + (d[2][2] + d[3][2]) + ((d[0][3] + d[1][3]) + (d[2][3] + d[3][3]));
        float* rb = red + (team * 2 + (it & 1)) * kTB * 16;
        if (tw == 1 && q < tb) {
          rb[q * 16 + g] = vlo;
          rb[q * 16 + 8 + g] = vhi;
        }
        bar_sync(kBarTeam0 + team, 2 * 32);
        if (tw == 0 && q < tb) {
          vlo += rb[q * 16 + g];
          vhi += rb[q * 16 + 8 + g];
          if (ok && !aborted(c)) {
            const float slo = c.hdr->scl[slot][rlo], shi = c.hdr->scl[slot][rhi];
            pair_epilogue(op, w, s, up ? g : rlo, rhi, q, vlo * slo, vhi * shi, dslot, dwt);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_n(&c.hdr->empty[slot], arrivals);
    }
    c.st += (uint32_t)nst;
  }

  // Pair epilogue, run by lane t for activation row t: v0, v1 are the dot
  // products of the pair's two weight rows r0, r1 (rows of stage s).
  __device__ __forceinline__ void pair_epilogue(int op, const int32_t* w, int s, int r0, int r1, int t, float v0,
                                                float v1, int dslot, float dwt) {
    const int l = w[F_LAYER];
    switch (op) {
      case OP_QKV_PROJ: {
        // RoPE in the epilogue, then the new K/V into the pool ("Tasks":
        // QKV_PROJ applies RoPE in-register before writing back); the row's
        // rotation by pos * base^(-dd/D) was tabulated for the step
        const int row = w[F_A0] + s * S::SR_H + r0;  // even: (row, row + 1) is a rotation pair
        const int b = t;
        const int head = row / S::D, dd = row - head * S::D;
        const int pos = sm.row_pos[b], page = sm.row_page[b];
        if (head < S::NQ + S::NKV) {
          const float2 cs = sm.rope_cs[b][dd / 2];
          const float x0 = v0 * cs.x - v1 * cs.y, x1 = v0 * cs.y + v1 * cs.x;
          v0 = x0;
          v1 = x1;
        }
        if (head < S::NQ) {
          *reinterpret_cast<float2*>(p.q + ((int64_t)b * S::NQ + head) * S::D + dd) = make_float2(v0, v1);
        } else if (pos >= 0) {
          const bool is_v = head >= S::NQ + S::NKV;
          const int g = head - S::NQ - (is_v ? S::NKV : 0);
          const uint32_t packed = (uint32_t)f_bf16(v0) | ((uint32_t)f_bf16(v1) << 16);
          *reinterpret_cast<uint32_t*>(p.kvnew + (((int64_t)b * 2 + (is_v ? 1 : 0)) * S::NKV + g) * S::D + dd) = packed;
          if (page < 0 || page >= p.num_pages) {
            record_error(p, ERR_PAGE, c.sm, where_of(w), pos / S::P, (uint32_t)page, (uint32_t)p.num_pages);
          } else {
            uint16_t* pool = is_v ? p.vpool : p.kpool;
            const int64_t o = ((((int64_t)l * p.num_pages + page) * S::NKV + g) * S::P + pos % S::P) * S::D + dd;
            *reinterpret_cast<uint32_t*>(pool + o) = packed;
          }
        }
        break;
      }
      case W_UP_TILE: {  // SiLU(gate) * up ("Tasks": the SiLU-and-multiply epilogue)
        constexpr MoePlan mp = gemv_plan_of<S, M>();
        const float act = v0 / (1.f + expf(-v0)) * v1;
        const int row = w[F_A0 + 2] + t;
        p.u[(int64_t)row * S::I + w[F_A0 + 1] * mp.up_tile + s * mp.up_half + r0] = act;
        break;
      }
      case OP_ROUTER_GEMM: {
        const int e = w[F_A0] + s * S::SR_H + r0;
        float* dst = p.rlog + ((int64_t)l * p.MB + t) * S::E + e;
        dst[0] = v0 + (p.rbias ? p.rbias[e] : 0.f);
        dst[1] = v1 + (p.rbias ? p.rbias[e + 1] : 0.f);
        break;
      }
      case OP_LM_HEAD: {
        const int v = w[F_A0] + s * S::SR_H + r0;
        *reinterpret_cast<float2*>(p.logits + (int64_t)t * p.V + v) = make_float2(v0, v1);
        break;
      }
      case OP_O_PROJ: {
        const int n = w[F_A0] + s * S::SR_O + r0;
        *reinterpret_cast<float2*>(p.opart + (((int64_t)(l & 1) * S::NKV + w[F_A0 + 2]) * p.MB + t) * S::H + n) =
            make_float2(v0, v1);
        break;
      }
      case W_DOWN_TILE: {  // weighted, into the (row b, slot j) of the output
        constexpr MoePlan mp = gemv_plan_of<S, M>();
        const int n = w[F_A0 + 1] * mp.dn_tile + s * mp.dn_rows + r0;
        *reinterpret_cast<float2*>(p.y + (int64_t)dslot * S::H + n) = make_float2(dwt * v0, dwt * v1);
        break;
      }
      default: break;
    }
  }

  // GEMV of at most kTB activation rows (decode at small batch).  The
  // consumer warps form four teams of two that take stages in turn, so four
  // stages are in process at once; within a stage each warp takes half of
  // the weight rows, two pairs at a time against the same activation loads,
  // and finishes each pair's epilogue itself (the RoPE pair for QKV, gate and
  // up rows for the MoE up/gate), so a stage needs no block-wide barrier.
  // One activation row has its own instantiation, without the second row's work.
  template <int K>
  __device__ __forceinline__ void gemv_item_teams(const int32_t* w, int SR, int total_rows, int ntok) {
    // one activation row is the decode case: its own instantiation, without
    // the second row's predicated work
    if (ntok <= 1) gemv_item_teams_tb<K, 1>(w, SR, total_rows, ntok);
    else gemv_item_teams_tb<K, kTB>(w, SR, total_rows, ntok);
  }
  static constexpr int kTeams = 4, kTeamWarps = kConsumerWarps / kTeams;
  // each warp of a team stands for its share of the arrivals a stage expects
  // (kConsumerWarps; two in the tensor-core builds, one per warp of the team)
  static constexpr int kTeamArrivals = mode_tc(M) ? 1 : kConsumerWarps / kTeamWarps;
  static_assert(kConsumerWarps % kTeams == 0 && F_A0 + 8 + 2 * kTB <= F_TASK, "teams; down-tile row fields");
  template <int K, int TB>
  __device__ __forceinline__ void gemv_item_teams_tb(const int32_t* w, int SR, int total_rows, int ntok) {
    constexpr int C = K / 8;
    constexpr int CPL = (C + 31) / 32;
    const int op = w[F_OP];
    const int nst = w[F_NSTAGE];
    const int tb = ntok;
    // epilogue inputs of lane t (activation row t), from the item (the
    // producer read them when it made the down tile)
    int dslot = 0;
    float dwt = 0.f;
    if (op == W_DOWN_TILE && lane < tb) {  // (constant indices: w stays in registers)
      dslot = lane == 0 ? w[F_A0 + 8] : w[F_A0 + 9];
      dwt = __int_as_float(lane == 0 ? w[F_A0 + 10] : w[F_A0 + 11]);
    }
    int32_t tag[4];
    x_tag(op, w, 0, tag);
    if (!(tag[0] == sm.xtag[0] && tag[1] == sm.xtag[1] && tag[2] == sm.xtag[2] && tag[3] == sm.xtag[3])) {
      if (!aborted(c)) load_x<K>(op, w, 0, tb);
      consumers_sync();
      if (ct == 0) {
        sm.xtag[0] = tag[0]; sm.xtag[1] = tag[1]; sm.xtag[2] = tag[2]; sm.xtag[3] = tag[3];
      }
    }
    const int team = cw / kTeamWarps, tw = cw % kTeamWarps;
    const bool up_pairs = op == W_UP_TILE;
    // x row t as [half][chunk][4]: lane's chunk c = lane + 32 j holds elements
    // 8c .. 8c+3 in half 0 and 8c+4 .. 8c+7 in half 1
    const uint32_t xs_a = smem_u32(sm.xs) + (uint32_t)lane * 16u;
    for (int s = team; s < nst; s += kTeams) {
      const uint32_t gs = c.st + (uint32_t)s;
      const int slot = gs % kStages;
      // The slot's previous use (stage s - kStages) may belong to another
      // team (kStages is not a multiple of kTeams): wait until it is released
      // first, so the parity wait below cannot match a phase two fills back.
      bool ok = s < kStages || mbar_wait(p, c, &c.hdr->empty[slot], ((gs / kStages) - 1) & 1);
      ok = __all_sync(FULL, ok && mbar_wait(p, c, &c.hdr->full[slot], (gs / kStages) & 1) && !aborted(c));
      const int rows = min(SR, total_rows - s * SR);
      const int npairs = rows / 2;
      // this warp's pairs [p0, p1): the first half of the stage's pairs, or the second
      const int per = (npairs + kTeamWarps - 1) / kTeamWarps;
      const int p0 = tw * per, p1 = min(npairs, p0 + per);
      const uint32_t st_a = smem_u32(stage(slot)) + (uint32_t)lane * 16u;
      if (ok) {
        for (int pr = p0; pr < p1; pr += 2) {
          // pairs pr and pr + 1 (the second repeats the first when absent)
          const int pq = pr + 1 < p1 ? pr + 1 : pr;
          int rr[4];
          rr[0] = up_pairs ? pr : 2 * pr;
          rr[1] = up_pairs ? pr + npairs : 2 * pr + 1;
          rr[2] = up_pairs ? pq : 2 * pq;
          rr[3] = up_pairs ? pq + npairs : 2 * pq + 1;
          // accumulators per row and activation row: even and odd elements
          float acc[4][TB][2];
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int t = 0; t < TB; ++t) acc[q][t][0] = acc[q][t][1] = 0.f;
          // unrolled by 4, not fully: the smaller loop body fetches better
          // (instruction fetch is one of this kernel's top stalls)
#pragma unroll 4
          for (int j = 0; j < CPL; ++j) {
            if (C % 32 == 0 || lane + 32 * j < C) {
              uint4 u[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) u[q] = lds128(st_a + (uint32_t)(rr[q] * K * 2 + j * 512));
#pragma unroll
              for (int t = 0; t < TB; ++t)
                if (TB == 1 || t < tb) {
                  const uint4 xa = lds128(xs_a + (uint32_t)((t * 2 * C + 32 * j) * 16));
                  const uint4 xb = lds128(xs_a + (uint32_t)((t * 2 * C + C + 32 * j) * 16));
#pragma unroll
                  for (int q = 0; q < 4; ++q) dot8_bf16(u[q], xa, xb, acc[q][t][0], acc[q][t][1]);
                }
            }
          }
          float v[4][TB];
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int t = 0; t < TB; ++t)
              if (TB == 1 || t < tb) v[q][t] = warp_sum(acc[q][t][0] + acc[q][t][1]);
          // lane t finishes the pairs for activation row t
          if (lane < tb && !aborted(c)) {
            const bool r1 = TB > 1 && lane == 1;
            pair_epilogue(op, w, s, rr[0], rr[1], lane, r1 ? v[0][TB - 1] : v[0][0], r1 ? v[1][TB - 1] : v[1][0],
                          dslot, dwt);
            if (pq != pr)
              pair_epilogue(op, w, s, rr[2], rr[3], lane, r1 ? v[2][TB - 1] : v[2][0], r1 ? v[3][TB - 1] : v[3][0],
                            dslot, dwt);
          }
        }
      }
      // the team's warps stand for the eight arrivals the stage expects
      __syncwarp();
      if (lane == 0) mbar_arrive_n(&c.hdr->empty[slot], kTeamArrivals);
    }
    c.st += (uint32_t)nst;
  }

  // --------------------------------------------------------- attention
  // Byte address of (token t, 16-byte chunk c16 of the head dims) in a KV page
  // stored as TMA tiles of (P tokens x 128 bytes) with the 128-byte swizzle.
  static __device__ __forceinline__ uint32_t kv_addr(uint32_t base, int t, int c16) {
    return base + (uint32_t)((c16 >> 3) * S::P * 128 + t * 128 + (((c16 & 7) ^ (t & 7)) << 4));
  }

  // One KV slice of one (row b, KV group g): its G query heads against the
  // keys in [t0, t1), as an unnormalised partial (running max in the log2
  // domain, sum, weighted values) -- "Tasks": ATTN_DECODE on a partial slice.
  // On tensor cores: per page, S = Q K^T with the heads as the MMA's rows
  // (padded to 16) and the warp's 8 tokens as its columns, then O += P V with
  // the warp's head dims as columns.  q and P enter as BF16 hi + lo pairs, so
  // the products keep fp32-level accuracy; K and V are BF16 as stored.
  __device__ __forceinline__ void attn(const int32_t* w) {
    constexpr int G = S::G, D = S::D, P = S::P, KS = D / 16, NT = D / 64;
    const int l = w[F_LAYER], b = w[F_A0], g = w[F_A0 + 1], t0 = w[F_A0 + 2], t1 = w[F_A0 + 3];
    const int pf = w[F_A0 + 4], slot_idx = w[F_A0 + 5], np = w[F_NSTAGE];
    // the row's new position (tabulated for the step at batch <= kTB)
    const int pos = b < p.B ? (p.B <= kTB ? sm.row_pos[b] : __ldg(p.seq_lens + b) - 1) : -1;
    const int qg = lane >> 2, qc = lane & 3;  // MMA fragment coordinates
    // The new token's K/V (written by the QKV tiles after the pool page was
    // read) replace its slot below; the slice that holds it loads them now,
    // in the same round as the queries.
    const bool has_new = pos >= t0 && pos < t1 && np > 0;
    uint4 kvn = make_uint4(0u, 0u, 0u, 0u);
    if (has_new && ct < 2 * D / 8) {
      const int which = ct / (D / 8), cc = ct % (D / 8);
      kvn = __ldcg(reinterpret_cast<const uint4*>(p.kvnew + (((int64_t)b * 2 + which) * S::NKV + g) * D) + cc);
    }
    // the group's queries, scaled by log2(e)/sqrt(D), split into BF16 hi + lo,
    // kept while (layer, b, g) repeats
    if (np > 0 && !(sm.qtag[0] == l && sm.qtag[1] == b && sm.qtag[2] == g)) {
      const float scale = 1.4426950408889634f / sqrtf((float)D);
      const float2* src = reinterpret_cast<const float2*>(p.q + ((int64_t)b * S::NQ + g * G) * D);
      for (int i = ct; i < 8 * D / 2; i += kConsumerThreads) {
        const int h = i / (D / 2), d2 = i - h * (D / 2);
        uint32_t hi = 0u, lo = 0u;
        if (h < G) {
          const float2 v = __ldcg(src + i);
          split_bf16x2(v.x * scale, v.y * scale, hi, lo);
        }
        *reinterpret_cast<uint32_t*>(&sm.qh[h][2 * d2]) = hi;
        *reinterpret_cast<uint32_t*>(&sm.ql[h][2 * d2]) = lo;
      }
      consumers_sync();
      if (ct == 0) {
        sm.qtag[0] = l; sm.qtag[1] = b; sm.qtag[2] = g;
      }
    }
    // ldmatrix rows of the Q fragments: head lane & 7, 16-byte chunk by lane >> 3
    const uint32_t qh_a = smem_u32(&sm.qh[lane & 7][8 * (lane >> 3)]);
    const uint32_t ql_a = smem_u32(&sm.ql[lane & 7][8 * (lane >> 3)]);
    float o[NT][4];  // this warp's NT tiles of 8 head dims
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    if (ct < G) {
      sm.am[ct] = -INFINITY;
      sm.al[ct] = 0.f;
    }
    const bool qk_warp = cw * 8 < P;  // this warp's 8 tokens exist in a page
    for (int k = 0; k < np; ++k) {
      int slot;
      const bool ok = __all_sync(FULL, stage_wait(slot) && !aborted(c));
      uint8_t* page = c.stages + (size_t)slot * kStageBytes;
      const uint32_t kb = smem_u32(page), vb = kb + (uint32_t)(NT * P * 128);
      const int page_t0 = (pf + k) * P;
      // the new token's K/V replace its slot: the pool page may predate the write
      if (has_new && pos >= page_t0 && pos < page_t0 + P) {
        const int sl = pos - page_t0;
        if (ok && ct < 2 * D / 8) {
          const int which = ct / (D / 8), cc = ct % (D / 8);
          const uint32_t a = kv_addr(which ? vb : kb, sl, cc);
          *reinterpret_cast<uint4*>(page + (a - kb)) = kvn;
          fence_proxy_async_smem();
        }
        consumers_sync();
      }
      // S = Q K^T for this warp's 8 tokens: Q's BF16 hi part in rows 0-7 of
      // the MMA and its lo part in rows 8-15 (one MMA takes both), even and
      // odd k-steps in separate accumulators (half the dependent chain)
      float sc[2] = {0.f, 0.f};
      if (ok && qk_warp) {
        const int tr = cw * 8 + (lane & 7);
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < KS; ks += 2) {
          uint32_t b0, b1, b2, b3, h0, h1, h2, h3, l0, l1, l2, l3;
          ldsm_x4(kv_addr(kb, tr, 2 * ks + (lane >> 3)), b0, b1, b2, b3);
          ldsm_x4(qh_a + ks * 32, h0, h1, h2, h3);
          ldsm_x4(ql_a + ks * 32, l0, l1, l2, l3);
          mma_bf16(sa, h0, l0, h1, l1, b0, b1);
          mma_bf16(sb, h2, l2, h3, l3, b2, b3);
        }
        sc[0] = (sa[0] + sa[2]) + (sb[0] + sb[2]);
        sc[1] = (sa[1] + sa[3]) + (sb[1] + sb[3]);
      }
      // this thread: head qg, tokens cw*8 + 2qc, +1
      const int tk = page_t0 + cw * 8 + 2 * qc;
      float s0 = (qk_warp && qg < G && tk >= t0 && tk < t1) ? sc[0] : -INFINITY;
      float s1 = (qk_warp && qg < G && tk + 1 >= t0 && tk + 1 < t1) ? sc[1] : -INFINITY;
      float mx = fmaxf(s0, s1);
      mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 2));
      if (qc == 0) sm.wred[cw][qg] = mx;
      consumers_sync();
      float pm = -INFINITY;
#pragma unroll
      for (int i = 0; i < kConsumerWarps; ++i) pm = fmaxf(pm, sm.wred[i][qg]);
      const float m_old = sm.am[qg % G];
      const float m_new = fmaxf(m_old, pm);
      const float p0 = (s0 == -INFINITY || m_new == -INFINITY) ? 0.f : exp2f(s0 - m_new);
      const float p1 = (s1 == -INFINITY || m_new == -INFINITY) ? 0.f : exp2f(s1 - m_new);
      float sum = p0 + p1;
      sum += __shfl_xor_sync(FULL, sum, 1);
      sum += __shfl_xor_sync(FULL, sum, 2);
      if (qc == 0) sm.wsum[cw][qg] = sum;
      if (qk_warp) {
        uint32_t hi, lo;
        split_bf16x2(p0, p1, hi, lo);
        *reinterpret_cast<uint32_t*>(&sm.ph[qg][cw * 8 + 2 * qc]) = hi;
        *reinterpret_cast<uint32_t*>(&sm.pl[qg][cw * 8 + 2 * qc]) = lo;
      }
      const float alpha = (m_old == -INFINITY) ? 0.f : exp2f(m_old - m_new);
      consumers_sync();
      if (cw == 0 && qc == 0 && qg < G) {
        float tot = 0.f;
#pragma unroll
        for (int i = 0; i < kConsumerWarps; ++i) tot += sm.wsum[i][qg];
        sm.al[qg] = sm.al[qg] * alpha + tot;
        sm.am[qg] = m_new;
      }
      // O += P V for this warp's head dims [8 NT cw, 8 NT (cw + 1))
      if (ok) {
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          o[n][0] *= alpha;
          o[n][1] *= alpha;
          o[n][2] *= alpha;
          o[n][3] *= alpha;
        }
#pragma unroll
        for (int kt = 0; kt < P / 16; ++kt) {
          uint32_t ah0 = 0u, ah2 = 0u, al0 = 0u, al2 = 0u;
          if (qg < G) {
            ah0 = *reinterpret_cast<const uint32_t*>(&sm.ph[qg][kt * 16 + 2 * qc]);
            ah2 = *reinterpret_cast<const uint32_t*>(&sm.ph[qg][kt * 16 + 8 + 2 * qc]);
            al0 = *reinterpret_cast<const uint32_t*>(&sm.pl[qg][kt * 16 + 2 * qc]);
            al2 = *reinterpret_cast<const uint32_t*>(&sm.pl[qg][kt * 16 + 8 + 2 * qc]);
          }
          const int tr = kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          // P's hi part in rows 0-7, its lo part in rows 8-15 (summed at the end)
          if (NT == 2) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(kv_addr(vb, tr, 2 * cw + (lane >> 4)), b0, b1, b2, b3);
            mma_bf16(o[0], ah0, al0, ah2, al2, b0, b1);
            mma_bf16(o[1], ah0, al0, ah2, al2, b2, b3);
          } else {
            uint32_t b0, b1;
            ldsm_x2_t(kv_addr(vb, tr, cw), b0, b1);
            mma_bf16(o[0], ah0, al0, ah2, al2, b0, b1);
          }
        }
      }
      stage_release(slot);
    }
    consumers_sync();
    if (aborted(c)) return;
    const int64_t base = ((int64_t)b * S::NKV + g) * p.max_slots + slot_idx;
    if (qg < G) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const int dcol = (NT * cw + n) * 8 + 2 * qc;
        *reinterpret_cast<float2*>(p.part_o + (base * G + qg) * D + dcol) =
            make_float2(o[n][0] + o[n][2], o[n][1] + o[n][3]);
      }
    }
    if (ct < G) {
      p.part_ml[(base * G + ct) * 2 + 0] = np > 0 ? sm.am[ct] : -INFINITY;
      p.part_ml[(base * G + ct) * 2 + 1] = np > 0 ? sm.al[ct] : 0.f;
    }
  }

  // Merge of the slice partials of (b, g): warp per head ("Tasks": ATTN_COMBINE).
  // Lanes read 32 slices' (max, sum) at once; the weighted values of a block
  // of slices are then loaded together, so a combine costs a few round trips.
  __device__ __forceinline__ void attn_combine(const int32_t* w) {
    constexpr int G = S::G, D = S::D, DPL = D / 32;
    const int l = w[F_LAYER], b = w[F_A0], g = w[F_A0 + 1];
    if constexpr (!kLean) {
      if (w[F_A0 + 3] >= 0) {  // one task per head
        attn_combine_one_head(l, b, g, w[F_A0 + 3]);
        return;
      }
    }
    if (b >= p.B || cw >= G) return;
    float o[DPL];
    combine_head(l, b, g, cw, o);
    const int64_t col = (int64_t)(g * G + cw) * D + lane * DPL;
    float* dst = p.attn_out + (int64_t)b * S::NQ * D + col;
#pragma unroll
    for (int i = 0; i < DPL; ++i) dst[i] = o[i];
    if constexpr (mode_tc(M) && DPL == 4) {
      store_hilo4(p.attnb + (int64_t)(2 * b) * S::NQ * D + col, p.attnb + (int64_t)(2 * b + 1) * S::NQ * D + col,
                  make_float4(o[0], o[1 % DPL], o[2 % DPL], o[3 % DPL]));
    } else if constexpr (mode_tc(M)) {
#pragma unroll
      for (int i = 0; i < DPL; ++i) {
        const uint16_t hi = f_bf16(o[i]);
        p.attnb[(int64_t)(2 * b) * S::NQ * D + col + i] = hi;
        p.attnb[(int64_t)(2 * b + 1) * S::NQ * D + col + i] = f_bf16(o[i] - bf16_f(hi));
      }
    }
  }

  // Head h of (b, g) by the whole block (few rows: the merge is on the path
  // from the last KV slice to the O projection).  Warp w merges a contiguous
  // block of the slices against its own running max, loading eight slices'
  // (max, sum) and values at once, so a block costs one round trip; the
  // eight partial merges meet in shared memory, taken in warp order.
  __device__ __forceinline__ void attn_combine_one_head(int l, int b, int g, int h) {
    constexpr int G = S::G, D = S::D, DPL = D / 32, J = 8;
    static_assert(kConsumerWarps * D <= kTB * xs_row<S>(), "the warps' partial sums fit the activation cache");
    // the activation cache holds the partial sums below: mark it empty
    // (read again only after the barrier that ends this item)
    if (ct == 0) sm.xtag[0] = -1;
    if (b >= p.B) return;
    const bool full = p.window == 0 || (l + 1) % p.full_period == 0;
    const int n = min(full ? slices_of(p, __ldg(p.seq_lens + b)) : p.n_static, p.max_slots);
    const int64_t base = ((int64_t)b * S::NKV + g) * p.max_slots;
    const int per = (n + kConsumerWarps - 1) / kConsumerWarps;
    const int j0 = cw * per, j1 = min(n, j0 + per);
    float m = -INFINITY, z = 0.f, acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
    for (int jb = j0; jb < j1; jb += J) {
      float2 ml[J];
      float o[J][DPL];
#pragma unroll
      for (int k = 0; k < J; ++k) {
        const int j = min(jb + k, j1 - 1);  // past the block: a repeated load, not used
        ml[k] = __ldcg(reinterpret_cast<const float2*>(p.part_ml + ((base + j) * G + h) * 2));
        const float* oj = p.part_o + ((base + j) * G + h) * D + lane * DPL;
        if (DPL == 4) {
          const float4 o4 = __ldcg(reinterpret_cast<const float4*>(oj));
          o[k][0] = o4.x; o[k][1 % DPL] = o4.y; o[k][2 % DPL] = o4.z; o[k][3 % DPL] = o4.w;
        } else {
#pragma unroll
          for (int i = 0; i < DPL; ++i) o[k][i] = __ldcg(oj + i);
        }
      }
      float mb = m;
#pragma unroll
      for (int k = 0; k < J; ++k)
        if (jb + k < j1 && ml[k].y > 0.f) mb = fmaxf(mb, ml[k].x);
      if (mb > m) {  // rescale what the warp has so far to the new max
        const float sc = exp2f(m - mb);
        z *= sc;
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] *= sc;
        m = mb;
      }
#pragma unroll
      for (int k = 0; k < J; ++k)
        if (jb + k < j1 && ml[k].y > 0.f) {
          const float cj = exp2f(ml[k].x - m);
          z = fmaf(cj, ml[k].y, z);
#pragma unroll
          for (int i = 0; i < DPL; ++i) acc[i] = fmaf(cj, o[k][i], acc[i]);
        }
    }
    float* red = sm.xs;  // [warp][D]
#pragma unroll
    for (int i = 0; i < DPL; ++i) red[cw * D + lane * DPL + i] = acc[i];
    if (lane == 0) {
      sm.red[cw] = z;
      sm.red[kConsumerWarps + cw] = m;
    }
    consumers_sync();
    if (ct < D) {
      float mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < kConsumerWarps; ++k)
        if (sm.red[k] > 0.f) mx = fmaxf(mx, sm.red[kConsumerWarps + k]);
      float zt = 0.f, a = 0.f;
#pragma unroll
      for (int k = 0; k < kConsumerWarps; ++k)
        if (sm.red[k] > 0.f) {
          const float sc = exp2f(sm.red[kConsumerWarps + k] - mx);
          zt = fmaf(sc, sm.red[k], zt);
          a = fmaf(sc, red[k * D + ct], a);
        }
      const float o = a / zt;
      const int64_t col = (int64_t)(g * G + h) * D + ct;
      p.attn_out[(int64_t)b * S::NQ * D + col] = o;
      if constexpr (mode_tc(M)) {
        const uint16_t hi = f_bf16(o);
        p.attnb[(int64_t)(2 * b) * S::NQ * D + col] = hi;
        p.attnb[(int64_t)(2 * b + 1) * S::NQ * D + col] = f_bf16(o - bf16_f(hi));
      }
    }
  }

  // Head h of (b, g) merged over the slices, by one warp: lane holds dims
  // [lane * DPL, lane * DPL + DPL).  The merge is on the path from the last
  // KV slice to the O projection, so its loads go out in as few rounds as
  // registers allow: every slice's (max, sum) together with the first CB
  // slices' partial outputs, then CB more slices per round.  The arithmetic
  // is the plain definition in slice order: the global max over the slices,
  // then acc = sum_j 2^(m_j - max) o_j and z = sum_j 2^(m_j - max) l_j.
  template <int DPL>
  __device__ __forceinline__ void combine_head(int l, int b, int g, int h, float (&out)[DPL]) {
    constexpr int G = S::G, D = S::D, MAXC = 4, CB = 16;
    static_assert(DPL == D / 32, "lane dims");
    const bool full = p.window == 0 || (l + 1) % p.full_period == 0;
    const int n = min(full ? slices_of(p, __ldg(p.seq_lens + b)) : p.n_static, p.max_slots);
    const int64_t base = ((int64_t)b * S::NKV + g) * p.max_slots;
    auto load_o = [&](int j, float (&o)[DPL]) {
      const float* oj = p.part_o + ((base + j) * G + h) * D + lane * DPL;
      if constexpr (DPL == 4) {
        const float4 o4 = __ldcg(reinterpret_cast<const float4*>(oj));
        o[0] = o4.x; o[1 % DPL] = o4.y; o[2 % DPL] = o4.z; o[3 % DPL] = o4.w;
      } else {
#pragma unroll
        for (int i = 0; i < DPL; ++i) o[i] = __ldcg(oj + i);
      }
    };
    float acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
    float z = 0.f, mx = -INFINITY;
    if (n <= 32 * MAXC) {
      // round 1: the (max, sum) of slices lane + 32k and the first CB slices' outputs
      float2 ml[MAXC];
#pragma unroll
      for (int k = 0; k < MAXC; ++k) {
        const int j = lane + 32 * k;
        ml[k] = j < n ? __ldcg(reinterpret_cast<const float2*>(p.part_ml + ((base + j) * G + h) * 2))
                      : make_float2(0.f, 0.f);
      }
      float o[CB][DPL];
#pragma unroll
      for (int k = 0; k < CB; ++k) load_o(min(k, n - 1), o[k]);
#pragma unroll
      for (int k = 0; k < MAXC; ++k)
        if (ml[k].y > 0.f) mx = fmaxf(mx, ml[k].x);
      mx = warp_max(mx);
      float cj[MAXC];
#pragma unroll
      for (int k = 0; k < MAXC; ++k) {
        cj[k] = ml[k].y > 0.f ? exp2f(ml[k].x - mx) : 0.f;
        z = fmaf(cj[k], ml[k].y, z);
      }
      static_assert(32 % CB == 0, "a round of slices lies in one register of cj");
      for (int j0 = 0; j0 < n; j0 += CB) {
        if (j0 > 0)  // the next round of CB slices
#pragma unroll
          for (int k = 0; k < CB; ++k) load_o(min(j0 + k, n - 1), o[k]);
        // slice j's coefficient sits in lane j % 32, register j / 32
        float cr = cj[0];
#pragma unroll
        for (int q = 1; q < MAXC; ++q)
          if (q == (j0 >> 5)) cr = cj[q];
#pragma unroll
        for (int k = 0; k < CB; ++k) {
          const float c = __shfl_sync(FULL, cr, (j0 + k) & 31);
          if (j0 + k < n)
#pragma unroll
            for (int i = 0; i < DPL; ++i) acc[i] = fmaf(c, o[k][i], acc[i]);
        }
      }
    } else {
      // many slices: the max first, then the slices in order, one at a time
      for (int j = lane; j < n; j += 32) {
        const float2 m2 = __ldcg(reinterpret_cast<const float2*>(p.part_ml + ((base + j) * G + h) * 2));
        if (m2.y > 0.f) mx = fmaxf(mx, m2.x);
      }
      mx = warp_max(mx);
      for (int j0 = 0; j0 < n; j0 += 32) {
        float c = 0.f;
        if (j0 + lane < n) {
          const float2 m2 = __ldcg(reinterpret_cast<const float2*>(p.part_ml + ((base + j0 + lane) * G + h) * 2));
          if (m2.y > 0.f) {
            c = exp2f(m2.x - mx);
            z = fmaf(c, m2.y, z);
          }
        }
        const int cnt = min(32, n - j0);
        for (int jj = 0; jj < cnt; ++jj) {
          const float cb = __shfl_sync(FULL, c, jj);
          float o[DPL];
          load_o(j0 + jj, o);
#pragma unroll
          for (int i = 0; i < DPL; ++i) acc[i] = fmaf(cb, o[i], acc[i]);
        }
      }
    }
    z = warp_sum(z);
    const float inv = 1.f / z;
#pragma unroll
    for (int i = 0; i < DPL; ++i) out[i] = acc[i] * inv;
  }

  // ------------------------------------------------------------- norm
  // Residual add + RMSNorm ("1. Reduce wave quantization": attention and MoE
  // rejoin only at the fused residual add + RMSNorm at the end of the layer).
  // Layer 0 starts from the embedding row; with the combine fused, the MoE
  // output of the previous layer is the sum of the row's K expert outputs,
  // which the down projection stored already weighted, one slot per (row, k).
  // Every operand is loaded with one round of independent 16-byte loads.
  // The residual entering layer l for row b -- the embedding at layer 0, else
  // the previous residual plus the attention partials plus the MoE output --
  // and its inverse RMS ("Residual + RMSNorm").  The residual buffer is kept
  // per layer parity, so layer l reads (l - 1) & 1 while its norm writes l & 1.
  template <int PER>
  __device__ __forceinline__ float resid_row(const int32_t* w, int l, int b, bool fused, float4 (&v)[PER]) {
    constexpr int H4 = S::H / 4;
#pragma unroll
    for (int k = 0; k < PER; ++k) v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (l == 0) {
      const int sl = __ldg(p.seq_lens + b);
      if ((sl < 1 || sl > p.max_ctx) && ct == 0) record_error(p, ERR_INDEX, c.sm, where_of(w), -1, (uint32_t)sl, (uint32_t)p.max_ctx);
      int tok = __ldg(p.tokens + b);
      if (tok < 0 || tok >= p.V) {
        if (ct == 0) record_error(p, ERR_INDEX, c.sm, where_of(w), -1, (uint32_t)tok, (uint32_t)p.V);
        tok = 0;
      }
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const int i4 = ct + k * kConsumerThreads;
        if (H4 % kConsumerThreads == 0 || i4 < H4) {
          const uint2 e = __ldg(reinterpret_cast<const uint2*>(p.emb + (int64_t)tok * S::H) + i4);
          v[k] = make_float4(bf16_lo(e.x), bf16_hi(e.x), bf16_lo(e.y), bf16_hi(e.y));
        }
      }
    } else {
      const float4* h4 = reinterpret_cast<const float4*>(p.h + ((int64_t)((l + 1) & 1) * p.MB + b) * S::H);
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const int i4 = ct + k * kConsumerThreads;
        if (H4 % kConsumerThreads == 0 || i4 < H4) {
          float4 parts[1 + S::NKV + S::K];
          int n = 0;
          parts[n++] = __ldcg(h4 + i4);
#pragma unroll
          for (int g = 0; g < S::NKV; ++g)
            parts[n++] = __ldcg(
                reinterpret_cast<const float4*>(p.opart + (((int64_t)((l + 1) & 1) * S::NKV + g) * p.MB + b) * S::H) + i4);
          if (fused) {
#pragma unroll
            for (int j = 0; j < S::K; ++j)
              parts[n++] = __ldcg(reinterpret_cast<const float4*>(p.y + ((int64_t)b * S::K + j) * S::H) + i4);
          } else {
            parts[n++] = __ldcg(reinterpret_cast<const float4*>(p.moe_out + (int64_t)b * S::H) + i4);
          }
          // residual + attention partials, then the MoE output summed on its own
          // (the same order as a separate MOE_COMBINE)
          float4 a = parts[0];
#pragma unroll
          for (int q = 1; q <= S::NKV; ++q) {
            a.x += parts[q].x; a.y += parts[q].y; a.z += parts[q].z; a.w += parts[q].w;
          }
          float4 m = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int q = 1 + S::NKV; q < 1 + S::NKV + S::K; ++q)
            if (q < n) {
              m.x += parts[q].x; m.y += parts[q].y; m.z += parts[q].z; m.w += parts[q].w;
            }
          a.x += m.x; a.y += m.y; a.z += m.z; a.w += m.w;
          v[k] = a;
        }
      }
    }
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < PER; ++k)
      ss = fmaf(v[k].x, v[k].x, fmaf(v[k].y, v[k].y, fmaf(v[k].z, v[k].z, fmaf(v[k].w, v[k].w, ss))));
    ss = warp_sum(ss);
    if (lane == 0) sm.red[cw] = ss;
    consumers_sync();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < kConsumerWarps; ++i) tot += sm.red[i];
    consumers_sync();  // sm.red is free again
    return 1.f / sqrtf(tot / (float)S::H + p.eps);
  }

  // This thread's float4s of a gain row (issued before the residual parts
  // are loaded, so that both arrive in the same round).
  template <int PER>
  __device__ __forceinline__ void load_gain(const float* gamma, float4 (&gm)[PER]) {
    constexpr int H4 = S::H / 4;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int i4 = ct + k * kConsumerThreads;
      gm[k] = (H4 % kConsumerThreads == 0 || i4 < H4) ? __ldg(reinterpret_cast<const float4*>(gamma) + i4)
                                                       : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }

  __device__ __forceinline__ void norm(const int32_t* w) {
    constexpr int H4 = S::H / 4, PER = (H4 + kConsumerThreads - 1) / kConsumerThreads;
    const int l = w[F_LAYER], b1 = min(w[F_A0 + 1], p.B);
    const bool final_norm = w[F_A0 + 2] != 0, fused = w[F_A0 + 3] != 0;
    // the gain row is loaded with the residual parts (one round of loads)
    float4 gms[PER];
    load_gain<PER>(final_norm ? p.gamma_f : p.gamma + (int64_t)l * S::H, gms);
    for (int b = w[F_A0]; b < b1; ++b) {
      float4 v[PER];
      const float inv_rms = resid_row<PER>(w, l, b, fused, v);
      float4* hout = reinterpret_cast<float4*>(p.h + ((int64_t)(l & 1) * p.MB + b) * S::H);
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const int i4 = ct + k * kConsumerThreads;
        if (H4 % kConsumerThreads == 0 || i4 < H4) {
          const float4 gm = gms[k], a = v[k];
          const float4 xv =
              make_float4(a.x * inv_rms * gm.x, a.y * inv_rms * gm.y, a.z * inv_rms * gm.z, a.w * inv_rms * gm.w);
          reinterpret_cast<float4*>(p.x + (int64_t)b * S::H)[i4] = xv;
          if constexpr (mode_tc(M))
            store_hilo4(p.xb + (int64_t)(2 * b) * S::H + 4 * i4, p.xb + (int64_t)(2 * b + 1) * S::H + 4 * i4, xv);
          if (!final_norm) hout[i4] = a;
          if (p.htrace) reinterpret_cast<float4*>(p.htrace + ((int64_t)l * p.MB + b) * S::H)[i4] = a;
        }
      }
    }
  }

  // A router task that computes the layer's RMSNorm itself (batch <= kTB):
  // the normalised rows go straight into the activation cache, in the layout
  // and with the tag the GEMV uses for the layer input.
  __device__ __forceinline__ void norm_into_cache(const int32_t* w) {
    constexpr int H4 = S::H / 4, PER = (H4 + kConsumerThreads - 1) / kConsumerThreads;
    const int l = w[F_LAYER];
    // a previous item of this SM left the same rows (uniform, as for the combine)
    if (sm.xtag[0] == 1 && sm.xtag[1] == 0 && sm.xtag[2] == 0 && sm.xtag[3] == l) return;
    float4* xs4 = reinterpret_cast<float4*>(sm.xs);
    float4 gms[PER];
    load_gain<PER>(p.gamma + (int64_t)l * S::H, gms);
    for (int b = 0; b < p.B; ++b) {
      float4 v[PER];
      const float inv_rms = resid_row<PER>(w, l, b, true, v);
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const int i4 = ct + k * kConsumerThreads;
        if (H4 % kConsumerThreads == 0 || i4 < H4) {
          const float4 gm = gms[k], a = v[k];
          // float4 i4 of the row goes to [half i4 % 2][chunk i4 / 2], as load_x places it
          xs4[b * H4 + (i4 & 1) * (H4 / 2) + (i4 >> 1)] =
              make_float4(a.x * inv_rms * gm.x, a.y * inv_rms * gm.y, a.z * inv_rms * gm.z, a.w * inv_rms * gm.w);
        }
      }
    }
    // the tag is read again within this item: publish it before the barrier
    if (ct == 0) {
      sm.xtag[0] = 1; sm.xtag[1] = 0; sm.xtag[2] = 0; sm.xtag[3] = l;
    }
    consumers_sync();
  }

  // The routing step of the last router task of a layer: count this task in;
  // the last one reads every router logit, runs the top-k and builds the MoE
  // queue, then signals the routing barrier itself.
  __device__ __forceinline__ void route_if_last(const int32_t* w) {
    // the block's logit stores, then one acquire-release count: the last
    // task sees every other task's logits
    consumers_sync();
    if (ct == 0) {
      const uint32_t old = atom_add_acq_rel(p.bars + w[F_A0 + 2], 1u);
      sm.flag = (old + 1u == (uint32_t)w[F_A0 + 3] && !aborted(c)) ? 1 : 0;
    }
    consumers_sync();
    if (!sm.flag) return;
    topk_rows(w[F_LAYER], 0, p.B, true);
    if (p.B == 1) {  // warp 0 finishes the row and releases the routing itself
      if (cw == 0) route_one_row(w[F_LAYER], p.bars + w[F_A0 + 4]);
      return;
    }
    consumers_sync();
    if (ct == 0) red_release_add(p.bars + w[F_A0 + 4], 1u);
  }

  // ------------------------------------------------------------ routing
  // Top-k of each row's router logits (higher logit first, lower expert id on
  // ties) and softmax weights over the selected logits ("Tasks": ROUTER_TOPK).
  __device__ __forceinline__ void topk(const int32_t* w) {
    const bool fin = w[F_A0 + 2] != 0;
    topk_rows(w[F_LAYER], w[F_A0], w[F_A0 + 1], fin);
    if (fin && p.B == 1 && cw == 0) route_one_row(w[F_LAYER], nullptr);  // the storer signals
  }
  // Logits as unsigned keys with the same order (finite inputs): a warp-wide
  // unsigned max then finds the largest logit in one reduction.
  static __device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  }
  static __device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
  }
  // One warp per row: K rounds of (max key over the warp, then the lowest
  // expert id holding it), written compactly -- this runs once per layer,
  // usually from a cold instruction cache.
  __device__ __forceinline__ void topk_rows(int l, int b0, int b_end, bool fin) {
    constexpr int E = S::E, K = S::K, PL = (E + 31) / 32;
    const int b1 = min(b_end, p.B);
    for (int b = b0 + cw; b < b1; b += kConsumerWarps) {
      uint32_t key[PL];
#pragma unroll
      for (int k = 0; k < PL; ++k) {
        const int e = lane + 32 * k;
        key[k] = e < E ? order_key(__ldcg(p.rlog + ((int64_t)l * p.MB + b) * E + e)) : 0u;
      }
#pragma unroll 1
      for (int j = 0; j < K; ++j) {
        uint32_t lk = 0u;
        uint32_t le = 0xffffffffu;
#pragma unroll
        for (int k = 0; k < PL; ++k)
          if (key[k] > lk) {
            lk = key[k];
            le = (uint32_t)(lane + 32 * k);
          }
        const uint32_t mk = __reduce_max_sync(FULL, lk);
        const uint32_t wi = __reduce_min_sync(FULL, lk == mk ? le : 0xffffffffu);
#pragma unroll
        for (int k = 0; k < PL; ++k)
          if ((uint32_t)(lane + 32 * k) == wi) key[k] = 0u;
        if (lane == 0) {
          sm.tk_id[cw][j] = (int32_t)wi;
          sm.tk_key[cw][j] = mk;
        }
      }
      __syncwarp();
      if (fin && p.B == 1) break;  // route_one_row finishes the row
      // softmax over the selected logits, lane j for choice j
      const float v0 = key_value(sm.tk_key[cw][0]);
      const float ej = lane < K ? expf(key_value(sm.tk_key[cw][lane < K ? lane : 0]) - v0) : 0.f;
      const float z = warp_sum(ej);
      if (lane < K) {
        const int id = sm.tk_id[cw][lane];
        p.topk_ids[((int64_t)l * p.MB + b) * K + lane] = id;
        p.topk_w[((int64_t)l * p.MB + b) * K + lane] = ej / z;
        sm.ids[b * K + lane] = id;
      }
      __syncwarp();
    }
    if (fin && p.B == 1) return;  // the caller runs route_one_row
    if (fin) {  // the one top-k task also builds the queues, from shared memory
      if (p.B > 1) consumers_sync();
      else __syncwarp();  // one row: warp 0 wrote the routing
      finalize(l, false);
    }
  }

  // The routing of a single row (decode at batch 1) after its top-k rounds,
  // by warp 0, lane j for choice j: the softmax weight, the rank of the
  // chosen expert among the chosen ids -- each has exactly one routed row, so
  // the rank is its place in the expert-ordered list -- and the queue record.
  // What the MoE branch reads is written first and released on `sig`; the
  // per-expert counts and offsets follow.
  __device__ __forceinline__ void route_one_row(int l, uint32_t* sig) {
    constexpr int E = S::E, K = S::K, PL = (E + 31) / 32;
    int my = 0x7fffffff, rank = 0;
    if (lane < K) {
      my = sm.tk_id[0][lane];
      if (my < 0 || my >= E) {
        record_error(p, ERR_INDEX, c.sm, kNowhere, -1, (uint32_t)my, E);
        my = 0;
      }
#pragma unroll
      for (int i = 0; i < K; ++i) rank += sm.tk_id[0][i] < my ? 1 : 0;
    }
    const float v0 = key_value(sm.tk_key[0][0]);
    const float ej = lane < K ? expf(key_value(sm.tk_key[0][lane < K ? lane : 0]) - v0) : 0.f;
    const float z = warp_sum(ej);
    int32_t* qt = queue_trace(l);
    if (lane < K) {
      p.topk_ids[(int64_t)l * p.MB * K + lane] = my;
      p.topk_w[(int64_t)l * p.MB * K + lane] = ej / z;
      reinterpret_cast<int4*>(p.act)[rank] = make_int4(my, rank, 1, 0);
      p.perm[rank] = lane;
      p.inv[lane] = rank;
      sm.ids[lane] = my;
      if (qt) {
        reinterpret_cast<int4*>(qt)[rank] = make_int4(my, rank, 1, 0);
        qt[5 * E + 1 + rank] = lane;
      }
    }
    if (lane == 0) *reinterpret_cast<int2*>(p.qlen) = make_int2(K, K);  // active experts, routed rows
    if (lane == 0 && qt) {
      qt[5 * E + 1 + p.MB * K] = K;
      qt[5 * E + 1 + p.MB * K + 1] = K;
    }
    __syncwarp();
    if (lane == 0 && sig) red_release_add(sig, 1u);
    // per-expert counts and offsets (outputs; nothing downstream waits on them)
#pragma unroll
    for (int k = 0; k < PL; ++k) {
      const int e = lane + 32 * k;
      int below = 0, chosen = 0;
#pragma unroll
      for (int i = 0; i < K; ++i) {
        const int id = sm.tk_id[0][i];
        below += id < e ? 1 : 0;
        chosen += id == e ? 1 : 0;
      }
      if (e < E) {
        p.ecount[(int64_t)l * E + e] = chosen;
        p.eoff[e] = below;
        if (qt) qt[4 * E + e] = below;
      }
    }
    if (lane == 0) p.eoff[E] = K;
    if (lane == 0 && qt) qt[5 * E] = K;
  }

  // This layer's record of the MoE queue trace, or null (see queue_trace_stride).
  __device__ __forceinline__ int32_t* queue_trace(int l) const {
    return p.qtrace ? p.qtrace + (int64_t)l * queue_trace_stride(S::E, p.MB * S::K) : nullptr;
  }

  // Per-expert counts and offsets, the expert-ordered row list (rows of an
  // expert by row b ascending) and the list of active experts, ascending
  // ("Tasks": ROUTE_FINALIZE generates the MoE GEMM work queue).  The queue of
  // the up/gate drain is (active expert a, tile t) for a ascending, t
  // ascending -- entry i is (list[i / tiles], i % tiles) -- and likewise for the
  // down drain, so the list is all the queue needs.  One warp does it, with
  // every lane owning a few experts' row bitmaps; nothing depends on atomics.
  __device__ __forceinline__ void finalize(int l, bool load_ids) {
    if (cw != 0) return;
    constexpr int E = S::E, K = S::K, PL = (E + 31) / 32;
    const int B = p.B, n = B * K;
    if (load_ids) {  // a separate task: the routing comes from global memory
      for (int i = lane; i < n; i += 32) {
        const int b = i / K;
        sm.ids[i] = __ldcg(p.topk_ids + ((int64_t)l * p.MB + b) * K + (i - b * K));
      }
      __syncwarp();
    }
    // each expert's rows as a bit mask (bit b: row b routes to it), the
    // warp's lanes taking every 32nd routed slot
    for (int e = lane; e < E; e += 32) sm.mask[e] = 0ull;
    __syncwarp();
    for (int i = lane; i < n; i += 32) {
      int e = sm.ids[i];
      if (e < 0 || e >= E) {
        record_error(p, ERR_INDEX, c.sm, kNowhere, -1, (uint32_t)e, E);
        e = 0;
      }
      atomicOr(&sm.mask[e], 1ull << (i / K));
    }
    __syncwarp();
    unsigned long long m[PL];
#pragma unroll
    for (int k = 0; k < PL; ++k) m[k] = lane * PL + k < E ? sm.mask[lane * PL + k] : 0ull;
    int cnt[PL], a[PL];
    int rs = 0, as = 0;
#pragma unroll
    for (int k = 0; k < PL; ++k) {
      cnt[k] = __popcll(m[k]);
      a[k] = cnt[k] > 0;
      rs += cnt[k];
      as += a[k];
    }
    int ri = rs, ai = as;  // inclusive scans over lanes
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int r2 = __shfl_up_sync(FULL, ri, d), a2 = __shfl_up_sync(FULL, ai, d);
      if (lane >= d) {
        ri += r2;
        ai += a2;
      }
    }
    int ro = ri - rs, ao = ai - as;
    int32_t* qt = queue_trace(l);
#pragma unroll
    for (int k = 0; k < PL; ++k) {
      const int e = lane * PL + k;
      if (e < E) {
        sm.mask[e] = m[k];
        sm.off[e] = ro;
        p.ecount[(int64_t)l * E + e] = cnt[k];
        p.eoff[e] = ro;
        if (a[k]) reinterpret_cast<int4*>(p.act)[ao] = make_int4(e, ro, cnt[k], 0);
        if (qt) {
          qt[4 * E + e] = ro;
          if (a[k]) reinterpret_cast<int4*>(qt)[ao] = make_int4(e, ro, cnt[k], 0);
        }
      }
      ro += cnt[k];
      ao += a[k];
    }
    if (lane == 31) {
      p.eoff[E] = ri;
      p.qlen[0] = ai;  // active experts
      p.qlen[1] = ri;  // routed rows
      if (qt) {
        qt[5 * E] = ri;
        qt[5 * E + 1 + p.MB * K] = ai;
        qt[5 * E + 1 + p.MB * K + 1] = ri;
      }
    }
    __syncwarp();
    for (int i = lane; i < n; i += 32) {
      const int b = i / K;
      int e = sm.ids[i];
      if (e < 0 || e >= E) e = 0;
      const int rank = __popcll(sm.mask[e] & ((1ull << b) - 1ull));
      const int row = sm.off[e] + rank;
      p.perm[row] = i;
      p.inv[i] = row;
      if (qt) qt[5 * E + 1 + row] = i;
    }
  }

  // expert-ordered copy of the routed rows ("Tasks": MOE_GATHER): a warp per
  // row, the warp's row indices read in one round, then each row in one
  // round of 16-byte loads
  __device__ __forceinline__ void gather(const int32_t* w) {
    constexpr int C = S::H / 4, PL = (C + 31) / 32, RW = 4;  // float4 per lane, rows per warp and round
    const int r0 = w[F_A0], r1 = min(r0 + w[F_A0 + 1], p.B * S::K);
    for (int rb = r0 + cw; rb < r1; rb += RW * kConsumerWarps) {
      int src[RW];
#pragma unroll
      for (int k = 0; k < RW; ++k) {
        const int r = rb + k * kConsumerWarps;
        const int pr = r < r1 ? __ldcg(p.perm + r) : 0;
        src[k] = (pr < 0 || pr / S::K >= p.B) ? 0 : pr / S::K;
      }
#pragma unroll 1
      for (int k = 0; k < RW; ++k) {
        const int r = rb + k * kConsumerWarps;
        if (r >= r1) break;
        const float4* x4 = reinterpret_cast<const float4*>(p.x + (int64_t)src[k] * S::H);
        float4 xv[PL];
#pragma unroll
        for (int q = 0; q < PL; ++q)
          if (C % 32 == 0 || lane + 32 * q < C) xv[q] = __ldcg(x4 + lane + 32 * q);
        [[maybe_unused]] float rs = 1.f;
        if constexpr (M == kModeTcFp8) {
          // the row's power-of-two scale into the E4M3 terms' range (its
          // inverse goes to the up/gate epilogue)
          float mx = 0.f;
#pragma unroll
          for (int q = 0; q < PL; ++q)
            if (C % 32 == 0 || lane + 32 * q < C)
              mx = fmaxf(mx, fmaxf(fmaxf(fabsf(xv[q].x), fabsf(xv[q].y)), fmaxf(fabsf(xv[q].z), fabsf(xv[q].w))));
          const int ke = e4m3_row_exponent(warp_max(mx));
          rs = ldexpf(1.f, ke);
          if (lane == 0) p.xg8s[r] = ldexpf(1.f, -ke);
        }
#pragma unroll
        for (int q = 0; q < PL; ++q) {
          const int cc = lane + 32 * q;
          if (C % 32 != 0 && cc >= C) continue;
          if constexpr (M == kModeTcFp8) {  // the FP8 expert tiles read the E4M3 term rows
            const float4 v = make_float4(xv[q].x * rs, xv[q].y * rs, xv[q].z * rs, xv[q].w * rs);
            store_e4m3_terms4(p.xg8 + (int64_t)kTcF8Terms * r * S::H + 4 * cc, S::H, v);
          } else if constexpr (M == kModeTc)  // the tcgen05 items read only the BF16 operand rows
            store_hilo4(p.xgb + (int64_t)(2 * r) * S::H + 4 * cc, p.xgb + (int64_t)(2 * r + 1) * S::H + 4 * cc, xv[q]);
          else
            reinterpret_cast<float4*>(p.xg + (int64_t)r * S::H)[cc] = xv[q];
        }
      }
    }
  }

  // weighted sum of each row's expert outputs ("Tasks": MOE_COMBINE); the
  // down projection stored each output already weighted in the row's slot
  __device__ __forceinline__ void moe_combine(const int32_t* w) {
    const int b1 = min(w[F_A0 + 1], p.B);
    for (int b = w[F_A0]; b < b1; ++b) {
      for (int i4 = ct; i4 < S::H / 4; i4 += kConsumerThreads) {
        float4 m = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < S::K; ++j) {
          const float4 y = __ldcg(reinterpret_cast<const float4*>(p.y + ((int64_t)b * S::K + j) * S::H) + i4);
          m.x += y.x; m.y += y.y; m.z += y.z; m.w += y.w;
        }
        reinterpret_cast<float4*>(p.moe_out + (int64_t)b * S::H)[i4] = m;
      }
    }
  }

  // ------------------------------------------------- tcgen05 GEMM items
  // An item of kModeTc: its kTcRows weight rows (M) against the activation
  // operand's tc_nb rows (N: every activation row as a hi row and a lo row),
  // K in k-blocks of kTcK, one stage each.  One thread issues the MMAs of a
  // stage as soon as its copies land, accumulating in TMEM (fp32), and hands
  // the stage back through tcgen05.commit (the stage's empty barrier counts
  // kConsumerWarps arrivals: one commit each).  A last commit marks the
  // accumulator complete; then every consumer warp reads its quarter of the
  // TMEM lanes (lane = weight row of the tile) for a share of the activation
  // rows (columns 2t and 2t + 1 hold hi and lo: their sum is row t's value)
  // and writes the outputs.  The next item's MMAs start after every warp has
  // read the accumulator (a block barrier between tcgen05 fences).
  __device__ __forceinline__ void tc_item(const int32_t* w) {
    const int op = w[F_OP];
    const int nst = w[F_NSTAGE], nkb = w[F_A0 + 13];
    // dense tiles' stages hold several k-blocks of their smaller weight boxes
    const uint32_t a_bytes = op == OP_ROUTER_GEMM                      ? kTcRouterRows * kTcK * 2
                             : (op == W_UP_TILE || op == W_DOWN_TILE) ? kTcMoeRows * kTcK * 2
                                                                      : kTcDenseRows * kTcK * 2;
    // FP8 expert tiles: E4M3 weights against the E4M3 term rows
    const bool f8 = M == kModeTcFp8 && (op == W_UP_TILE || op == W_DOWN_TILE);
    const int nb = f8 ? p.tc_nb8 : p.tc_nb;
    const int kps = tc_kblocks_per_stage(a_bytes, nb);
    const uint32_t bbytes = (uint32_t)nb * kTcK * 2;
    if (ct == 0) {
      tc_fence_after();
      // one MMA's K in descriptor units: 32 bytes (16 BF16 or 32 FP8 values),
      // four MMAs per 128-byte k-block
      constexpr uint32_t kDescK = 32 / 16;
      const uint32_t idesc = f8 ? tc_idesc_e4m3(kTcRows, nb) : tc_idesc_bf16(kTcRows, nb);
      for (int st = 0; st < nst; ++st) {
        const uint32_t gs = c.st + (uint32_t)st;
        const int slot = (int)(gs % kStages);
        if (!mbar_wait(p, c, &c.hdr->full[slot], (gs / kStages) & 1)) break;
        const uint32_t a = smem_u32(stage(slot));
        for (int j = 0; j < kps && st * kps + j < nkb; ++j) {
          const uint64_t ad = tc_desc_sw128(a + j * a_bytes), bd = tc_desc_sw128(a + kTcABytes + j * bbytes);
          if (M == kModeTcFp8 && f8) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc_mma_f8(tmem, ad + (uint64_t)(kDescK * k), bd + (uint64_t)(kDescK * k), idesc, (st | j | k) != 0);
          } else {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc_mma_bf16(tmem, ad + (uint64_t)(kDescK * k), bd + (uint64_t)(kDescK * k), idesc, (st | j | k) != 0);
          }
        }
        // the stage goes back to the producer once these MMAs have read it (in
        // these builds a stage's empty barrier takes two arrivals)
        tc_commit(&c.hdr->empty[slot]);
        tc_commit(&c.hdr->empty[slot]);
      }
      tc_commit(&c.hdr->acc_full);
    }
    c.st += (uint32_t)nst;
    const bool ok = mbar_wait(p, c, &c.hdr->acc_full, acc_phase);
    acc_phase ^= 1u;
    tc_fence_after();
    if (__all_sync(FULL, ok && !aborted(c))) tc_epilogue(w, op);
    tc_fence_before();
    consumers_sync();
  }

  // The accumulator of a tcgen05 item to its outputs: this warp's TMEM lanes
  // (weight rows 32 q .. 32 q + 31 of the tile, q = the warp's index in the
  // CTA modulo 4) for every other chunk of 8 activation rows (the two warps of
  // a quarter take alternate chunks).
  __device__ __forceinline__ void tc_epilogue(const int32_t* w, int op) {
    const int l = w[F_LAYER];
    const int q = (int)((threadIdx.x >> 5) & 3), half = cw >> 2;
    const int r = 32 * q + lane;  // this thread's row of the tile
    const bool moe = op == W_UP_TILE || op == W_DOWN_TILE;
    const int ntok = moe ? w[F_A0 + 3] : p.B;
    const int nrows = moe ? kTcMoeRows : w[F_A0 + 1];
    if (r >= ((nrows + 31) & ~31)) return;  // a warp quarter of unused MMA rows (uniform per warp)
    if constexpr (M == kModeTcFp8) {
      if (moe) {
        tc_epilogue_f8(w, op, l, q, half, r, ntok);
        return;
      }
    }
    constexpr MoePlan mp = S::mptc;
    for (int j = half; 8 * j < ntok; j += 2) {
      float c16[16];
      tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(16 * j), c16);
      float v[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) v[t] = c16[2 * t] + c16[2 * t + 1];
      switch (op) {
        case OP_QKV_PROJ: {
          // rows (2i, 2i + 1) sit in neighbouring lanes: the even lane rotates the pair
          float vp[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) vp[t] = __shfl_xor_sync(FULL, v[t], 1);
          // the chunk's positions, then their pages: two rounds of loads for 8 rows
          int pos[8], page[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) pos[t] = 8 * j + t < ntok ? __ldg(p.seq_lens + 8 * j + t) - 1 : -1;
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const int lp = pos[t] / S::P;
            page[t] = pos[t] >= 0 && lp < p.max_pages ? __ldg(p.block_tables + (int64_t)(8 * j + t) * p.max_pages + lp) : -1;
          }
          if ((lane & 1) == 0 && r < nrows) {
            const int row = w[F_A0] + r;
            const int head = row / S::D, dd = row - head * S::D;
#pragma unroll
            for (int t = 0; t < 8; ++t)
              if (8 * j + t < ntok) qkv_out(w, l, 8 * j + t, pos[t], page[t], head, dd, v[t], vp[t]);
          }
          break;
        }
        case OP_ROUTER_GEMM:
          if (r < nrows) {
            const int e = w[F_A0] + r;
            const float bias = p.rbias ? p.rbias[e] : 0.f;
#pragma unroll
            for (int t = 0; t < 8; ++t)
              if (8 * j + t < ntok) p.rlog[((int64_t)l * p.MB + 8 * j + t) * S::E + e] = v[t] + bias;
          }
          break;
        case OP_LM_HEAD:
          if (r < nrows)
#pragma unroll
            for (int t = 0; t < 8; ++t)
              if (8 * j + t < ntok) p.logits[(int64_t)(8 * j + t) * p.V + w[F_A0] + r] = v[t];
          break;
        case OP_O_PROJ:
          if (r < nrows)
#pragma unroll
            for (int t = 0; t < 8; ++t)
              if (8 * j + t < ntok)
                p.opart[(((int64_t)(l & 1) * S::NKV + w[F_A0 + 2]) * p.MB + 8 * j + t) * S::H + w[F_A0] + r] = v[t];
          break;
        case W_UP_TILE: {
          // lanes 0-15 of the warp hold gate rows 16 q .. 16 q + 15, lanes 16-31 the
          // same up rows: SiLU(gate) * up ("Tasks": the SiLU-and-multiply epilogue)
          float up[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) up[t] = __shfl_down_sync(FULL, v[t], 16);
          if (lane < 16 && r < nrows) {
            const int col = w[F_A0 + 1] * mp.up_tile + 16 * q + lane;
#pragma unroll
            for (int t = 0; t < 8; ++t)
              if (8 * j + t < ntok) {
                const int row = w[F_A0 + 2] + 8 * j + t;  // expert-ordered routed row
                const float act = v[t] / (1.f + expf(-v[t])) * up[t];
                p.u[(int64_t)row * S::I + col] = act;
                const uint16_t hi = f_bf16(act);
                p.ub[((int64_t)2 * row) * S::I + col] = hi;
                p.ub[((int64_t)2 * row + 1) * S::I + col] = f_bf16(act - bf16_f(hi));
              }
          }
          break;
        }
        case W_DOWN_TILE: {
          // weighted, into the (row b, slot j) the routed row belongs to: the
          // chunk's slots, then their weights (two rounds of loads for 8 rows)
          const int n = w[F_A0 + 1] * mp.dn_tile + r;
          int slot[8];
          float wt[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            slot[t] = 8 * j + t < ntok ? __ldcg(p.perm + w[F_A0 + 2] + 8 * j + t) : 0;
            if (slot[t] < 0 || slot[t] >= p.B * S::K) slot[t] = 0;  // only after a failed step
          }
#pragma unroll
          for (int t = 0; t < 8; ++t) wt[t] = __ldcg(p.topk_w + (int64_t)l * p.MB * S::K + slot[t]);
#pragma unroll
          for (int t = 0; t < 8; ++t)
            if (8 * j + t < ntok) p.y[(int64_t)slot[t] * S::H + n] = wt[t] * v[t];
          break;
        }
        default: break;
      }
    }
  }

  // The accumulator of an FP8 expert tile (kModeTcFp8): columns
  // kTcF8Terms t + j hold the products with term j of routed row t, so row t's
  // value is their sum scaled by 16^-j, times the weight row's scale (E4M3 code
  // times the row scale is the weight) and, for an up/gate tile, the inverse
  // of the gathered row's scale.  Chunks of 4 routed rows (16 columns), the
  // two warps of a lane quarter taking alternate chunks.  The up/gate epilogue
  // writes the SwiGLU activations as the down tiles' E4M3 term rows (unscaled:
  // a value beyond 448 in magnitude fails the step with ERR_RANGE).
  __device__ __forceinline__ void tc_epilogue_f8(const int32_t* w, int op, int l, int q, int half, int r, int ntok) {
    constexpr MoePlan mp = S::mptc8;
    static_assert(kTcF8Terms == 4, "four term columns per routed row: 4 rows per 16-column load");
    const int64_t le = (int64_t)l * S::E + w[F_A0];
    const bool up_tile = op == W_UP_TILE;
    // this lane's weight row: gate row 16 q + lane (lanes 0-15) or the same up
    // row (lanes 16-31) of an up/gate tile; down row r of a down tile
    const int col = w[F_A0 + 1] * mp.up_tile + 16 * q + (lane & 15);
    const int n = w[F_A0 + 1] * mp.dn_tile + r;
    const float scale = up_tile ? __ldg((lane < 16 ? p.sg : p.su) + le * S::I + col) : __ldg(p.sd + le * S::H + n);
    bool bad = false;
    for (int j = half; 4 * j < ntok; j += 2) {
      float c16[16];
      tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(16 * j), c16);
      float v[4];
#pragma unroll
      for (int t = 0; t < 4; ++t)
        v[t] = scale * (c16[4 * t] + 0.0625f * (c16[4 * t + 1] + 0.0625f * (c16[4 * t + 2] + 0.0625f * c16[4 * t + 3])));
      if (up_tile) {
        float xs[4];  // the gathered rows' inverse scales
#pragma unroll
        for (int t = 0; t < 4; ++t) xs[t] = 4 * j + t < ntok ? __ldcg(p.xg8s + w[F_A0 + 2] + 4 * j + t) : 0.f;
        float upv[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          v[t] *= xs[t];
          upv[t] = __shfl_down_sync(FULL, v[t], 16);
        }
        if (lane < 16) {
#pragma unroll
          for (int t = 0; t < 4; ++t)
            if (4 * j + t < ntok) {
              const int row = w[F_A0 + 2] + 4 * j + t;  // expert-ordered routed row
              float act = v[t] / (1.f + expf(-v[t])) * upv[t];
              p.u[(int64_t)row * S::I + col] = act;
              bad |= !(fabsf(act) <= 448.f);
              uint8_t* dst = p.u8 + (int64_t)kTcF8Terms * row * S::I + col;
#pragma unroll
              for (int k = 0; k < kTcF8Terms; ++k) {
                const uint32_t code = f_e4m3x2(act, 0.f) & 0xffu;
                dst[(int64_t)k * S::I] = (uint8_t)code;
                act = (act - e4m3_f(code)) * 16.f;
              }
            }
        }
      } else {
        int slot[4];
        float wt[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          slot[t] = 4 * j + t < ntok ? __ldcg(p.perm + w[F_A0 + 2] + 4 * j + t) : 0;
          if (slot[t] < 0 || slot[t] >= p.B * S::K) slot[t] = 0;  // only after a failed step
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) wt[t] = __ldcg(p.topk_w + (int64_t)l * p.MB * S::K + slot[t]);
#pragma unroll
        for (int t = 0; t < 4; ++t)
          if (4 * j + t < ntok) p.y[(int64_t)slot[t] * S::H + n] = wt[t] * v[t];
      }
    }
    if (bad) record_error(p, ERR_RANGE, c.sm, where_of(w), col, 0u, 448u);
  }

  // One QKV rotation pair (rows dd, dd + 1 of head `head`) of activation row
  // b: RoPE by pos * base^(-dd/D) (angle reduced modulo 2 pi in double,
  // then sin/cos in float) on q and k; q to its buffer, k and v to the pool.
  __device__ __forceinline__ void qkv_out(const int32_t* w, int l, int b, int pos, int page, int head, int dd, float v0,
                                          float v1) {
    if (head < S::NQ + S::NKV) {
      const double ang = (double)pos * sm.rope_theta[dd / 2];
      const double red = ang - 6.283185307179586 * rint(ang * 0.15915494309189535);
      float s0, c0;
      sincosf((float)red, &s0, &c0);
      const float r0 = v0 * c0 - v1 * s0, r1 = v0 * s0 + v1 * c0;
      v0 = r0;
      v1 = r1;
    }
    if (head < S::NQ) {
      *reinterpret_cast<float2*>(p.q + ((int64_t)b * S::NQ + head) * S::D + dd) = make_float2(v0, v1);
    } else if (pos >= 0) {
      const bool is_v = head >= S::NQ + S::NKV;
      const int g = head - S::NQ - (is_v ? S::NKV : 0);
      const uint32_t packed = (uint32_t)f_bf16(v0) | ((uint32_t)f_bf16(v1) << 16);
      *reinterpret_cast<uint32_t*>(p.kvnew + (((int64_t)b * 2 + (is_v ? 1 : 0)) * S::NKV + g) * S::D + dd) = packed;
      if (page < 0 || page >= p.num_pages) {
        record_error(p, ERR_PAGE, c.sm, where_of(w), pos / S::P, (uint32_t)page, (uint32_t)p.num_pages);
      } else {
        uint16_t* pool = is_v ? p.vpool : p.kpool;
        const int64_t o = ((((int64_t)l * p.num_pages + page) * S::NKV + g) * S::P + pos % S::P) * S::D + dd;
        *reinterpret_cast<uint32_t*>(pool + o) = packed;
      }
    }
  }

  __device__ __forceinline__ void execute(const int32_t* w) {
    if constexpr (mode_tc(M)) {
      switch (w[F_OP]) {
        case W_UP_TILE:
        case W_DOWN_TILE:
          if (w[F_A0 + 3] <= kTB) break;  // an expert with one or two rows: the GEMV below
          tc_item(w);
          return;
        case OP_QKV_PROJ:
        case OP_LM_HEAD:
        case OP_O_PROJ:
          tc_item(w);
          return;
        case OP_ROUTER_GEMM:
          tc_item(w);
          if (w[F_A0 + 5]) route_if_last(w);
          return;
        default: break;
      }
    }
    // above kTB rows (any-batch mode only) the two-row GEMV; FP8 / FP4
    // experts take their tensor-core GEMVs
    constexpr bool any_batch = M == kModeAnyBatch;
    switch (w[F_OP]) {
      case OP_ROUTER_GEMM:
        if (w[F_A0 + 7] && p.B <= kTB) norm_into_cache(w);
        if (!any_batch || p.B <= kTB) gemv_item_teams<S::H>(w, S::SR_H, w[F_A0 + 1], p.B);
        else if constexpr (any_batch) gemv_item<S::H>(w, S::SR_H, w[F_A0 + 1], p.B);
        if (w[F_A0 + 5]) route_if_last(w);
        break;
      case OP_QKV_PROJ:
      case OP_LM_HEAD:
        if (w[F_OP] == OP_QKV_PROJ && w[F_A0 + 7] && p.B <= kTB) norm_into_cache(w);
        if (!any_batch || p.B <= kTB) gemv_item_teams<S::H>(w, S::SR_H, w[F_A0 + 1], p.B);
        else if constexpr (any_batch) gemv_item<S::H>(w, S::SR_H, w[F_A0 + 1], p.B);
        break;
      case OP_O_PROJ:
        if (!any_batch || p.B <= kTB) gemv_item_teams<S::G * S::D>(w, S::SR_O, w[F_A0 + 1], p.B);
        else if constexpr (any_batch) gemv_item<S::G * S::D>(w, S::SR_O, w[F_A0 + 1], p.B);
        break;
      case W_UP_TILE:
        if constexpr (mode_fp4(M)) {
          if (w[F_A0 + 3] <= 1) gemv_item_fp4<S::H, 1>(w, w[F_A0 + 3]);
          else gemv_item_fp4<S::H, kTB>(w, w[F_A0 + 3]);
        } else if constexpr (mode_fp8(M) || M == kModeTcFp8) {
          constexpr MoePlan m8 = gemv_plan_of<S, M>();
          if (w[F_A0 + 3] <= 1) gemv_item_fp8<S::H, 1>(w, 2 * m8.up_half, w[F_A0 + 3]);
          else gemv_item_fp8<S::H, kTB>(w, 2 * m8.up_half, w[F_A0 + 3]);
        } else {
          constexpr MoePlan mg = gemv_plan_of<S, M>();
          if (!any_batch || w[F_A0 + 3] <= kTB)
            gemv_item_teams<S::H>(w, 2 * mg.up_half, 2 * mg.up_half * mg.up_stages, w[F_A0 + 3]);
          else if constexpr (any_batch)
            gemv_item<S::H>(w, 2 * mg.up_half, 2 * mg.up_half * mg.up_stages, w[F_A0 + 3]);
        }
        break;
      case W_DOWN_TILE:
        if constexpr (mode_fp4(M)) {
          if (w[F_A0 + 3] <= 1) gemv_item_fp4<S::I, 1>(w, w[F_A0 + 3]);
          else gemv_item_fp4<S::I, kTB>(w, w[F_A0 + 3]);
        } else if constexpr (mode_fp8(M) || M == kModeTcFp8) {
          constexpr MoePlan m8 = gemv_plan_of<S, M>();
          if (w[F_A0 + 3] <= 1) gemv_item_fp8<S::I, 1>(w, m8.dn_rows, w[F_A0 + 3]);
          else gemv_item_fp8<S::I, kTB>(w, m8.dn_rows, w[F_A0 + 3]);
        } else {
          constexpr MoePlan mg = gemv_plan_of<S, M>();
          if (!any_batch || w[F_A0 + 3] <= kTB) gemv_item_teams<S::I>(w, mg.dn_rows, mg.dn_tile, w[F_A0 + 3]);
          else if constexpr (any_batch) gemv_item<S::I>(w, mg.dn_rows, mg.dn_tile, w[F_A0 + 3]);
        }
        break;
      case W_ATTN: attn(w); break;
      case OP_ATTN_COMBINE: attn_combine(w); break;
      case OP_RESID_NORM: norm(w); break;
      // tasks of unfused schedules: not in the lean build
      case OP_ROUTER_TOPK: if constexpr (!kLean) topk(w); break;
      case OP_ROUTE_FINALIZE: if constexpr (!kLean) finalize(w[F_LAYER], true); break;
      case OP_MOE_GATHER: if constexpr (!kLean) gather(w); break;
      case OP_MOE_COMBINE: if constexpr (!kLean) moe_combine(w); break;
      default: break;  // NOP, CLAIM_END: only the signal
    }
  }

  // kModeTc: TMEM columns of the accumulator (the MMA's N is at most kTcMaxN)
  static constexpr uint32_t kTcCols = 128;
  static_assert(kTcMaxN <= (int)kTcCols, "the accumulator's columns");

  // kModeTc, after the last item: every MMA this CTA issued has completed
  // (one more commit, waited for with the usual time limit), then the TMEM
  // goes back -- also after a failed step, so the SM's TMEM is free again.
  __device__ __forceinline__ void tc_release() {
    if (ct == 0) {
      tc_commit(&c.hdr->tc_drain);
      const int64_t t0 = gtimer();
      while (!mbar_try_wait(&c.hdr->tc_drain, 0) && gtimer() - t0 < p.watchdog_ns) {
      }
    }
    tc_fence_before();
    consumers_sync();
    if (cw == 0) {
      tc_fence_after();
      tmem_dealloc(tmem, kTcCols);
    }
  }

  __device__ __forceinline__ void run() {
    // per-CTA set-up: the RoPE frequencies and empty activation caches
    for (int i = ct; i < S::D / 2; i += kConsumerThreads)
      sm.rope_theta[i] = pow((double)p.rope_base, -(double)(2 * i) / (double)S::D);
    if (ct < 4) sm.xtag[ct] = sm.qtag[ct] = -1;
    if constexpr (mode_tc(M)) {
      if (cw == 0) tmem_alloc(&c.hdr->tmem_addr, kTcCols);
      tc_fence_before();
    }
    consumers_sync();
    if constexpr (mode_tc(M)) {
      tc_fence_after();
      tmem = c.hdr->tmem_addr;
    }
    // at batch <= kTB the rows' rotations and KV pages hold for every layer:
    // computed once here, as the QKV epilogue would (angle reduced modulo
    // 2 pi in double, then sin/cos in float)
    if (p.B <= kTB) {
      for (int i = ct; i < p.B * (S::D / 2); i += kConsumerThreads) {
        const int b = i / (S::D / 2), k = i - b * (S::D / 2);
        const int pos = __ldg(p.seq_lens + b) - 1;
        const double ang = (double)pos * sm.rope_theta[k];
        const double red = ang - 6.283185307179586 * rint(ang * 0.15915494309189535);
        float s0, c0;
        sincosf((float)red, &s0, &c0);
        sm.rope_cs[b][k] = make_float2(c0, s0);
        if (k == 0) {
          const int lp = pos / S::P;
          sm.row_pos[b] = pos;
          sm.row_page[b] = (pos >= 0 && lp < p.max_pages) ? __ldg(p.block_tables + (int64_t)b * p.max_pages + lp) : -1;
        }
      }
      consumers_sync();
    }
    // thread 0 remembers a few counters it has already seen reach a count
    int cbar[4] = {-1, -1, -1, -1};
    uint32_t cval[4] = {0, 0, 0, 0};
    int crr = 0;
    auto seen = [&](int bar, uint32_t tgt) -> bool {
      if (bar < 0 || tgt == 0) return true;
      bool hit = false;
#pragma unroll
      for (int k = 0; k < 4; ++k) hit |= cbar[k] == bar && cval[k] >= tgt;
      return hit;
    };
    auto remember = [&](int bar, uint32_t tgt) {
      if (bar < 0 || tgt == 0) return;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (k == crr) {
          cbar[k] = bar;
          cval[k] = tgt;
        }
      crr = (crr + 1) & 3;
    };
    // an item's two waits, read together; counters seen complete are skipped
    auto wait_cached = [&](int b0, uint32_t t0, int b1, uint32_t t1, const int32_t* w) -> bool {
      const bool s0 = seen(b0, t0), s1 = seen(b1, t1);
      if (s0 && s1) return true;
      if (!wait_counters(p, c, s0 ? -1 : b0, t0, s1 ? -1 : b1, t1, where_of(w))) return false;
      if (!s0) remember(b0, t0);
      if (!s1) remember(b1, t1);
      return true;
    };
    uint32_t n_items = 0;
    for (;;) {
      const int slot = c.wk % kWorkRing;
      bool ok = mbar_wait(p, c, &c.hdr->wfull[slot], (c.wk / kWorkRing) & 1);
      int32_t w[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) w[k] = c.hdr->work[slot][k];
      // a claim end is only a signal: each thread hands it on without the
      // block barrier (every thread arrives after its earlier items, so the
      // storer still publishes it after them); the decision is uniform
      if (ok && w[F_OP] == W_CLAIM_END && w[F_SEQ] == (int32_t)c.wk && !aborted(c)) {
        ++c.wk;
        mbar_arrive(&c.hdr->done[slot]);
        continue;
      }
      const int64_t t_pop = (ct == 0 && (p.trace || p.stats)) ? gtimer() : 0;
      if (ct == 0) {
        p.prog[c.sm * 8 + 0] = n_items;
        p.prog[c.sm * 8 + 1] = (uint32_t)(w[F_OP] & 0xff) | ((uint32_t)(w[F_LAYER] & 0xff) << 8) |
                               ((uint32_t)(w[F_TASK] & 0xffff) << 16);
        p.prog[c.sm * 8 + 2] = c.st;
      }
      if (ok && ct == 0) {
        const uint32_t tgt0 = (uint32_t)(w[F_TGT0] == TGT_DYN_SPLITS
                                             ? (w[F_A0] < p.B ? slices_of(p, __ldg(p.seq_lens + w[F_A0])) : 0)
                                             : w[F_TGT0]);
        ok = wait_cached(w[F_WAIT0], tgt0, w[F_WAIT1], (uint32_t)w[F_TGT1], w);
      }
      if (ok && w[F_SEQ] != (int32_t)c.wk) {
        if (ct == 0) record_error(p, ERR_RING, c.sm, where_of(w), -2, (uint32_t)w[F_SEQ], c.wk);
        c.hdr->abort = 1;
        ok = false;
      }
      const int64_t t_go = (ct == 0 && (p.trace || p.stats)) ? gtimer() : 0;
      if (bar_or(kBarConsumers, kConsumerThreads, !ok || aborted(c))) return;
      ++c.wk;
      if (w[F_OP] == W_EXIT) {
        if (p.stats && ct == 0) {
          uint64_t* st = p.stats + (int64_t)c.sm * kStats;
          st[0] = c.stat[0];
          st[1] = c.stat[1];
          st[2] = c.stat[2];
          st[3] = n_items;
        }
        return;
      }
      execute(w);
      if (ct == 0 && (p.trace || p.stats)) {
        const int64_t t_end = gtimer();
        c.stat[0] += t_go - t_pop;
        c.stat[2] += t_end - t_go;
        if (p.trace && (int)n_items < p.trace_cap) {
          // record: popped, waits done, end (ns), and op | layer << 8 | task << 16 | a0 << 40
          uint64_t* r = p.trace + ((int64_t)c.sm * p.trace_cap + n_items) * 4;
          r[0] = (uint64_t)t_pop;
          r[1] = (uint64_t)t_go;
          r[2] = (uint64_t)t_end;
          r[3] = (uint64_t)(w[F_OP] & 0xff) | ((uint64_t)(w[F_LAYER] & 0xff) << 8) |
                 ((uint64_t)(uint32_t)(w[F_TASK] & 0xffffff) << 16) |
                 ((uint64_t)(uint32_t)(w[F_A0] & 0xffffff) << 40);
        }
      }
      ++n_items;
      // hand the item to the storer, which publishes it ("Storer: signal output barriers")
      mbar_arrive(&c.hdr->done[slot]);
    }
  }
};

// ======================================================================
// storer
// ======================================================================
// Publishes each finished item: after every consumer has arrived on the
// slot's `done` barrier (their outputs are written), one release add per
// signalled counter, then the slot goes back to the producer.
static __device__ void storer(const Params& p, Ctx& c) {
  if ((threadIdx.x & 31) != 0) return;
  Hdr* H = c.hdr;
  for (;;) {
    const int slot = c.wk % kWorkRing;
    const uint32_t par = (c.wk / kWorkRing) & 1;
    if (!mbar_wait(p, c, &H->wfull[slot], par)) return;
    const int op = H->work[slot][F_OP], sig0 = H->work[slot][F_SIG0], sig1 = H->work[slot][F_SIG1];
    if (H->work[slot][F_SEQ] != (int32_t)c.wk) {
      record_error(p, ERR_RING, c.sm, kNowhere, -3, (uint32_t)H->work[slot][F_SEQ], c.wk);
      H->abort = 1;
      return;
    }
    if (op == W_EXIT) return;
    if (!mbar_wait(p, c, &H->done[slot], par)) return;
    if (sig0 >= 0) red_release_add(p.bars + sig0, 1u);
    if (sig1 >= 0) red_release_add(p.bars + sig1, 1u);
    mbar_arrive(&H->wempty[slot]);
    ++c.wk;
    p.prog[c.sm * 8 + 6] = c.wk;
  }
}

template <class S, int M>
__global__ void __launch_bounds__(kThreads, 1) mk_persistent(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  // the 128-byte TMA swizzle of the KV pages is laid out from a 1024-byte
  // aligned stage base
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) record_error(p, ERR_SMEM_ALIGN, (int)blockIdx.x, kNowhere, -1, smem_u32(smem), 1024u);
    return;
  }
  static_assert(sizeof(Hdr) % 16 == 0 && alignof(Scratch<S>) <= 16, "scratch alignment");
  Hdr* hdr = reinterpret_cast<Hdr*>(smem + (size_t)kStages * kStageBytes);
  Scratch<S>* scr = reinterpret_cast<Scratch<S>*>(smem + (size_t)kStages * kStageBytes + sizeof(Hdr));
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&hdr->full[i], 1);
      // the tcgen05 build hands a stage back with one arrival (a commit of the
      // MMAs that read it, or one thread after the block's last read)
      mbar_init(&hdr->empty[i], mode_tc(M) ? 2 : kConsumerWarps);
    }
    for (int i = 0; i < kDescRing; ++i) {
      mbar_init(&hdr->dfull[i], 1);
      mbar_init(&hdr->dempty[i], 1);
    }
    for (int i = 0; i < kWorkRing; ++i) {
      mbar_init(&hdr->wfull[i], 1);
      mbar_init(&hdr->wempty[i], 1);
      mbar_init(&hdr->done[i], kConsumerThreads);
    }
    mbar_init(&hdr->acc_full, 1);
    mbar_init(&hdr->tc_drain, 1);
    hdr->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  Ctx c{hdr, smem, (int)blockIdx.x, 0u, 0u, {0, 0, 0, 0}};
  const int warp = threadIdx.x / 32;
  if (warp == 0) {
    controller(p, c);
  } else if (warp == 1) {
    Producer<S, M> pr{p, c, 0ull};
    pr.run();
  } else if (warp == 2) {
    storer(p, c);
  } else {
    const int ct = threadIdx.x - 96;
    Consumer<S, M> cs{p, c, *scr, ct, ct / 32, ct & 31};
    cs.run();
    if constexpr (mode_tc(M)) cs.tc_release();
  }
}

}  // namespace dev
}  // namespace mk
