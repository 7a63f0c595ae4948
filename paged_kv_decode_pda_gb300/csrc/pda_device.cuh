// Device-side primitives for the sm_103a decode path: mbarrier with bounded
// waits, 1-D bulk (TMA) copies, ldmatrix / movmatrix, warp MMA, fp8 and f16
// packing. All inline PTX is hand-written for this library.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace pda {

// Device status word: 0 = healthy. A kernel that gives up on a bounded wait
// ORs a code in here; pda_query_device_status reads and clears it. (The
// library is a single translation unit, so the definition lives here.)
__device__ unsigned int g_status = 0u;

enum : unsigned int {
  kStatusFullWaitTimeout = 1u << 0,   // consumer waited too long for a page fill
  kStatusEmptyWaitTimeout = 1u << 1,  // producer waited too long for a free ring slot
  kStatusDrainTimeout = 1u << 2,      // copies still in flight at exit after the limit
  kStatusTestWaitTimeout = 1u << 3,   // pda_test_bounded_wait gave up (expected)
  kStatusBadSlot = 1u << 4,           // reshape_and_cache saw a slot past the pool (skipped)
  kStatusMergeWaitTimeout = 1u << 5,  // persistent decode: consumer warps never met to merge a unit
  kStatusBadBlock = 1u << 6,          // decode with the block check on: a block id outside the pool
};

// Limit on any single barrier wait. Healthy waits last microseconds; the
// limit only bounds a wait that can no longer finish.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for the phase with the given parity to complete, for at most
// limit_ns. Returns false (without recording anything) on timeout or when
// *abort becomes nonzero; the caller records the reason.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort,
                                                  unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0u) {
      if (abort != nullptr && *abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) return false;
    }
  }
}

// Named barrier over `nthreads` threads that also ORs a predicate across
// them: every participant gets the same result.
__device__ __forceinline__ int named_barrier_or(int id, int nthreads, int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred), "r"(id), "r"(nthreads)
      : "memory");
  return r;
}

// ------------------------------------------------------------ bulk copies

// 1-D bulk copy global -> shared, completing `bytes` of transaction count on
// `bar`. dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 16-byte asynchronous copy global -> shared (L2 only, both addresses 16-byte
// aligned), tracked by cp_async_arrive_noinc.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// One arrival on `bar` once every cp.async this thread issued has landed.
// .noinc: the arrival is part of the count the barrier was initialised with.
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// 4-D tiled tensor copy global -> shared through a tensor map in kernel
// parameter space, completing its bytes on `bar`.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

// Four rows of a 2-D tensor map (box: one row of the map's width) in one
// copy: rows r0..r3 from column 0 land one after another at dst.
__device__ __forceinline__ void tma_gather4_rows(uint32_t dst, const CUtensorMap* map, int r0, int r1, int r2, int r3,
                                                 uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
      : "memory");
}

// Fetch a kernel-parameter tensor map's descriptor ahead of its first copy.
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// --------------------------------------------------------- warp fragments

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// As ldsm_x4, each 8x8 b16 matrix transposed on the way to registers.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// D += A(16x16, f16, row) * B(16x8, f16, col), fp32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two e4m3 bytes (low 16 bits of x) -> f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_lo_to_f16x2(uint32_t x) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(r) : "r"(x));
  return r;
}
// Two e4m3 bytes (high 16 bits of x) -> f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_hi_to_f16x2(uint32_t x) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, hi;\n\t}" : "=r"(r) : "r"(x));
  return r;
}

// (lo, hi) fp32 -> f16x2 with lo in the low half, round to nearest even.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two fp32 -> e4m3x2 (hi in the upper byte), round to nearest even,
// saturating finite (|x| > 448 and infinities give +-448; NaN stays NaN).
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Programmatic dependent launch: a kernel launched as the programmatic
// dependent of the previous one waits here until that kernel has finished
// and its memory writes are visible; the previous kernel lets it launch
// early with grid_dependents_launch().
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Thread-block clusters. cluster_sync: every thread of every CTA of the
// cluster arrives (releasing its earlier shared-memory writes at cluster
// scope) and waits for all the others (acquiring theirs). mapa_cluster: the
// address of the same shared-memory location in the cluster's CTA `rank`.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t mapa_cluster(uint32_t addr, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ float2 ld_cluster_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}

// 8-byte shared-memory load (8-byte aligned address).
__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 ld_nc_v2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

// bf16 pair (x = lo | hi << 16) -> fp32 pair, exact.
__device__ __forceinline__ float bf16lo_f32(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi_f32(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// f16 pair (x = lo | hi << 16) -> fp32 pair, exact.
__device__ __forceinline__ float f16lo_f32(uint32_t x) {
  return __half2float(__ushort_as_half((unsigned short)(x & 0xFFFFu)));
}
__device__ __forceinline__ float f16hi_f32(uint32_t x) { return __half2float(__ushort_as_half((unsigned short)(x >> 16))); }

// 2^n as a normal binary32 value, n in [-126, 127] (built from its exponent bits).
__device__ __forceinline__ float exp2_int(int n) { return __uint_as_float((uint32_t)(n + 127) << 23); }

}  // namespace pda
