// Shared device helpers for the Grok-1 GQA attention kernels (sm_103a only):
// inline-PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor), tcgen05
// (TMEM alloc / MMA / ld / st / commit), warp-level mma.sync, and bf16 packing.
//
// Every wait on an mbarrier is bounded: after GROK_WAIT_CYCLES clock cycles it
// records GROK_DEV_TIMEOUT in the caller's status word, raises the CTA's abort
// flag and returns false, so a kernel never hangs and never traps.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "grok_attn.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ != 1030)
#error "this library is written for sm_103a only"
#endif

namespace grok {

constexpr int kQHeads = GROK_N_Q_HEADS;
constexpr int kKVHeads = GROK_N_KV_HEADS;
constexpr int kGroup = kQHeads / kKVHeads;  // 6 query heads per KV head
constexpr int kD = GROK_HEAD_DIM;

// 1/sqrt(128) (attn_output_multiplier) and the soft cap 30.
constexpr float kMult = 0.08838834764831845f;
constexpr float kCap = 30.0f;
constexpr float kLog2e = 1.4426950408889634f;
// Softmax weight of a capped logit c relative to the fixed reference c = 30:
//   p = exp(c - 30) = 2^(30 log2(e) (tanh(y) - 1)),  y = s * mult / 30.
constexpr float kY = kMult / kCap;
constexpr float kT = kCap * kLog2e;

#ifndef GROK_WAIT_CYCLES
#define GROK_WAIT_CYCLES (4000000000LL)  // ~2 s at 2 GHz
#endif

// ----------------------------------------------------------------------------
// status word
__device__ __forceinline__ void report(int32_t* status, int32_t code) {
  if (status) atomicOr(status, code);
}

// ----------------------------------------------------------------------------
// KV-cache addressing. Contiguous: cache [B][Tmax][8][128], row (b, key).
// Paged: a pool [n_pages][GROK_PAGE_TOKENS][8][128] and a block table
// [B][max_pages] of page ids; key `key` of sequence b is row key % 128 of page
// table[b][key / 128]. As TMA coordinates: (row, b) contiguous, (page * 128 +
// key % 128, 0) paged. A page id outside [0, n_pages) reports
// GROK_DEV_BAD_PAGE and resolves to page 0 (a load stays in bounds; callers
// that store check kv_page_ok first).
struct PageMap {
  const int32_t* table;  // nullptr: contiguous cache
  int max_pages;
  int n_pages;
};

__device__ __forceinline__ bool kv_page_ok(const PageMap& pm, int b, int key) {
  if (!pm.table) return true;
  const int pg = __ldg(pm.table + (size_t)b * pm.max_pages + (key / GROK_PAGE_TOKENS));
  return pg >= 0 && pg < pm.n_pages;
}

__device__ __forceinline__ void kv_coord(const PageMap& pm, int b, int key, int& row, int& bc, int32_t* status) {
  if (!pm.table) {
    row = key;
    bc = b;
    return;
  }
  int pg = __ldg(pm.table + (size_t)b * pm.max_pages + (key / GROK_PAGE_TOKENS));
  if (pg < 0 || pg >= pm.n_pages) {
    report(status, GROK_DEV_BAD_PAGE);
    pg = 0;
  }
  row = pg * GROK_PAGE_TOKENS + key % GROK_PAGE_TOKENS;
  bc = 0;
}

// ----------------------------------------------------------------------------
// shared-memory addresses, mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity. Returns false (after
// recording a timeout and raising *abort) if the wait gives up after
// `limit` clock cycles, or as soon as another thread of the CTA has raised
// *abort.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, volatile int* abort,
                                              int32_t* status, long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > limit) {
      report(status, GROK_DEV_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          int32_t* status) {
  return mbar_wait_for(bar, parity, abort, status, GROK_WAIT_CYCLES);
}

// ----------------------------------------------------------------------------
// TMA
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// TMA store of a shared-memory box into a 4-d tensor, as a bulk async group of
// the issuing thread (coordinates must not be negative; rows past the tensor's
// extent are not written).
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* src, int c0, int c1, int c2,
                                             int c3) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The thread's committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// The thread's committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Generic-proxy shared-memory writes become visible to the async proxy (TMA, tensor cores).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ----------------------------------------------------------------------------
// tcgen05 (5th-generation tensor core, tensor memory)
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
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

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on *bar when every tcgen05.mma issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, M x N tile.
// b_mn_major = 1 when B's N dimension is the contiguous one.
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N, int b_mn_major) {
  return (1u << 4)                      // D format: f32
         | (1u << 7)                    // A format: bf16
         | (1u << 10)                   // B format: bf16
         | (0u << 15)                   // A K-major
         | (uint32_t(b_mn_major) << 16) // B major
         | (uint32_t(N >> 3) << 17)     // N / 8
         | (uint32_t(M >> 4) << 24);    // M / 16
}

// Shared-memory matrix descriptor for a 128-byte-swizzled tile (1024-byte aligned atoms).
__device__ __forceinline__ uint64_t make_sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFF);
  d |= uint64_t((lbo_bytes >> 4) & 0x3FFF) << 16;
  d |= uint64_t((sbo_bytes >> 4) & 0x3FFF) << 32;
  d |= uint64_t(1) << 46;  // descriptor version (sm_100 family)
  d |= uint64_t(2) << 61;  // swizzle: 128B
  return d;
}

// 32 lanes x 32 bit, 32 consecutive columns: thread i of the warp gets lane (base + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Wait for outstanding TMEM loads and tie the destination registers to the
// wait, so the compiler cannot move their uses above it.
__device__ __forceinline__ void tmem_wait_ld_dep(uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
        "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
        "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]),
        "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
        "+r"(r[30]), "+r"(r[31])
      :
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ----------------------------------------------------------------------------
// special-function-unit approximations (PTX)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Softmax weight relative to the fixed reference logit 30 (see kY, kT above),
// fast form: two special-function operations, tanh (absolute error measured
// below 8e-6 on sm_103, i.e. at most ~2.4e-4 relative in the weight) and ex2.
__device__ __forceinline__ float capped_weight(float s) {
  const float t = tanh_approx(s * kY);
  return ex2_approx(fmaf(t, kT, -kT));
}

// Precise form (~1e-6 relative): 30 (tanh(y) - 1) = -60 / (1 + e^(2y)), so
// p = 2^(-2 kT / (1 + 2^(2 y log2 e))) with three special-function operations.
__device__ __forceinline__ float capped_weight_precise(float s) {
  const float u = ex2_approx(s * (2.0f * kY * kLog2e));
  return ex2_approx((-2.0f * kT) * rcp_approx(1.0f + u));
}

// ----------------------------------------------------------------------------
// packed fp32 pairs: the sm_100-family f32x2 add/sub/mul/fma do two lanes' worth
// of IEEE single-precision work (same rounding as the scalar forms) in one issue
// slot. A pair lives in a 64-bit register: first element in the low half.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// 2^x for a pair of x in [-126, 0] on the FMA pipe instead of the special-
// function unit: x = j + f with j the nearest integer (rounded by adding
// 1.5 * 2^23, so j lands in the low mantissa bits of the sum) and f in
// [-1/2, 1/2]; 2^f from a degree-4 polynomial fitted here for relative error
// on [-1/2, 1/2] (weighted least squares refined toward equal ripple, then
// rounded to fp32: maximum relative error 2.7e-6 including the fp32 Horner
// steps); 2^j added to the exponent field. A NaN input need not give NaN.
__device__ __forceinline__ void exp2_poly_f2(uint64_t x, float& y0, float& y1) {
  const uint64_t big = f2_pack(12582912.0f, 12582912.0f);
  const uint64_t t = f2_add(x, big);
  const uint64_t f = f2_sub(x, f2_sub(t, big));
  uint64_t q = f2_fma(f2_pack(0x1.3997ca0p-7f, 0x1.3997ca0p-7f), f, f2_pack(0x1.ca14400p-5f, 0x1.ca14400p-5f));
  q = f2_fma(q, f, f2_pack(0x1.ec06da0p-3f, 0x1.ec06da0p-3f));
  q = f2_fma(q, f, f2_pack(0x1.62e0dc0p-1f, 0x1.62e0dc0p-1f));
  q = f2_fma(q, f, f2_pack(0x1.ffffe80p-1f, 0x1.ffffe80p-1f));
  float t0, t1, q0, q1;
  f2_unpack(t, t0, t1);
  f2_unpack(q, q0, q1);
  y0 = __uint_as_float(__float_as_uint(q0) + (__float_as_uint(t0) << 23));
  y1 = __uint_as_float(__float_as_uint(q1) + (__float_as_uint(t1) << 23));
}

// One lane of a converged warp (the same lane every time it is called).
__device__ __forceinline__ bool elect_one() {
  uint32_t e;
  asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(e));
  return e != 0;
}

// ----------------------------------------------------------------------------
// bf16 packing: cvt.rn.bf16x2.f32 d, a, b puts a in the upper half, b in the lower.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
// fp16 packing: cvt.rn.f16x2.f32 d, a, b puts a in the upper half, b in the lower.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Split fp32 pair (a, b) into bf16 hi + lo parts: a = hi_a + lo_a to ~2^-16 relative.
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(a, b);
  lo = pack_bf16x2(a - bf16lo_to_f32(hi), b - bf16hi_to_f32(hi));
}

// ----------------------------------------------------------------------------
// warp-level mma.sync m16n8k16 (bf16 in, fp32 accumulate) and ldmatrix
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t saddr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(saddr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t saddr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(saddr));
}

// Byte offset of element (row, col) in a [rows][64] bf16 tile written by TMA
// with 128-byte swizzle (tile base 1024-byte aligned): 16-byte chunk index is
// XORed with row % 8.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t col) {
  return row * 128u + ((((col >> 3) ^ (row & 7u)) & 7u) << 4) + ((col & 7u) << 1);
}

}  // namespace grok
