// tcgen05 / TMA / mbarrier helpers shared by the prefill attention kernels
// (prefill_tc.cu): thin inline-PTX wrappers, each one instruction or a
// bounded wait. M = 128 throughout (one CTA, cta_group::1).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

namespace {

constexpr int kTcM = 128;          // MMA rows (query rows of a work item)
constexpr int kSpin = 1 << 22;     // polls before a wait gives up

__device__ __forceinline__ uint32_t t_smem(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void t_bar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void t_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void t_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// waits for completion number k (0, 1, ...) of the barrier's phases; false
// if it gave up (the abort flag is then raised for everyone)
__device__ __forceinline__ bool t_wait(uint32_t bar, int k, volatile int *abort_flag) {
  const uint32_t parity = static_cast<uint32_t>(k) & 1u;
  for (int i = 0; i < kSpin; ++i) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred q;\nmbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n"
        "selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if ((i & 63) == 63 && *abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}
// whether completion number k of the barrier's phases has happened (one
// test, no wait)
__device__ __forceinline__ bool t_test(uint32_t bar, int k) {
  uint32_t done;
  asm volatile(
      "{\n.reg .pred q;\nmbarrier.test_wait.parity.shared::cta.b64 q, [%1], %2;\n"
      "selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(static_cast<uint32_t>(k) & 1u)
      : "memory");
  return done != 0;
}
// the same, by every lane of a warp, with one result for the warp (so the
// warp-collective TMEM accesses that follow are never reached by part of it)
__device__ __forceinline__ bool t_wait_warp(uint32_t bar, int k, volatile int *abort_flag) {
  return __all_sync(0xffffffffu, t_wait(bar, k, abort_flag));
}
// bounded wait that ignores the abort flag (used to drain the tensor core
// before the TMEM is released)
__device__ __forceinline__ void t_wait_drain(uint32_t bar) {
  for (int i = 0; i < kSpin; ++i) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred q;\nmbarrier.try_wait.parity.shared::cta.b64 q, [%1], 0;\n"
        "selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(done)
        : "r"(bar)
        : "memory");
    if (done) return;
  }
}
__device__ __forceinline__ void t_tma_1d(uint32_t dst, const CUtensorMap *tm, int x, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.1d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2}], [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(bar)
      : "memory");
}
// pulls one box of a 4-D tensor map into L2 only (no destination, no barrier)
__device__ __forceinline__ void t_prefetch_4d(const CUtensorMap *tm, int x, int y, int z, int w) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(tm)),
               "r"(x), "r"(y), "r"(z), "r"(w)
               : "memory");
}
__device__ __forceinline__ void t_tma_4d(uint32_t dst, const CUtensorMap *tm, int x, int y, int z,
                                         int w, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void t_tma_3d(uint32_t dst, const CUtensorMap *tm, int x, int y, int z,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
// shared-memory matrix descriptor: SW128 atoms, version 1
__device__ __forceinline__ uint64_t t_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}
// instruction descriptor, kind::f16: f32 accumulator, bf16 A and B, A
// K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1), M = 128
__host__ __device__ constexpr uint32_t t_idesc(int N, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(kTcM >> 4) << 24);
}
__device__ __forceinline__ void t_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                      uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void t_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void t_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void t_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void t_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void t_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]));
}
__device__ __forceinline__ void t_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void t_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// 2^x on the MUFU unit (the PTX approximate instruction, subnormal results
// flushed to zero: they are below what the bf16 P can hold anyway)
// max of three (one instruction on sm_100 and later)
__device__ __forceinline__ float t_max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// (d0, d1) = (a0, a1) * b + c, one packed instruction, each lane rounded as fmaf
__device__ __forceinline__ void t_fma2(float &d0, float &d1, float a0, float a1, float b, float c) {
  asm("{\n.reg .b64 ra, rb, rc, rd;\nmov.b64 ra, {%2, %3};\nmov.b64 rb, {%4, %4};\n"
      "mov.b64 rc, {%5, %5};\nfma.rn.f32x2 rd, ra, rb, rc;\nmov.b64 {%0, %1}, rd;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
// (s0, s1) += (a0, a1), one packed instruction
__device__ __forceinline__ void t_add2(float &s0, float &s1, float a0, float a1) {
  asm("{\n.reg .b64 rs, ra;\nmov.b64 rs, {%0, %1};\nmov.b64 ra, {%2, %3};\n"
      "add.rn.f32x2 rs, rs, ra;\nmov.b64 {%0, %1}, rs;\n}"
      : "+f"(s0), "+f"(s1)
      : "f"(a0), "f"(a1));
}
__device__ __forceinline__ float t_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t t_pack(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

}  // namespace
