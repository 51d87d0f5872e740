// Device-side building blocks for the CSA kernels (sm_103a):
//  - the cache byte layout (see include/csa.h, FORMAT),
//  - FP4 / FP8 encoders written in integer arithmetic (RNE, saturating),
//  - inline-PTX wrappers for mbarrier, TMA, bulk copies and tcgen05.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/csa.h"

namespace csa {

// ---- layout ------------------------------------------------------------------
constexpr int D = CSA_D, DI = CSA_DI, TOPK = CSA_TOPK, WIN = CSA_WINDOW;
constexpr int PAGE = CSA_PAGE_ENTRIES;
constexpr int KV_PAGE = CSA_KV_PAGE_BYTES, KV_SCALE_OFF = 16384;
constexpr int IDX_PAGE = CSA_IDX_PAGE_BYTES, IDX_GROUP = 544;   // 8-entry groups: 512 B data + 32 B scales

// Byte offsets inside an indexer page: data byte k of slot e, scale byte b of slot e.
__host__ __device__ constexpr int idx_data_off(int e, int k) {
  return IDX_GROUP * (e >> 3) + 128 * (k >> 4) + 16 * (e & 7) + (k & 15);
}
__host__ __device__ constexpr int idx_scale_off(int e, int b) { return IDX_GROUP * (e >> 3) + 512 + 4 * (e & 7) + b; }

// Status word at the head of the workspace (csa_check_device_status).
struct DeviceStatus {
  uint32_t flags;
  uint32_t pad[63];
};
constexpr size_t kStatusBytes = 256;

__device__ __forceinline__ void raise_flag(uint32_t* status, uint32_t f) {
  if (status) atomicOr(status, f);
}

// ---- scalar codecs --------------------------------------------------------------
// e2m1: nearest of {0,.5,1,1.5,2,3,4,6}; midpoints go to the even code
// (0.25->0, 0.75->1.0, 1.25->1.0, 1.75->2, 2.5->2, 3.5->4, 5->4); > 5 -> 6.
// The sign bit follows the input's sign bit (so -0.1 -> 0x8).
__device__ __forceinline__ uint32_t e2m1_rne(float v) {
  const uint32_t sign = (__float_as_uint(v) >> 28) & 8u;
  const float a = fabsf(v);
  uint32_t m = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) +
               (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
  return sign | m;
}

// E4M3 ("fn"): round to nearest even on the fp32 bit pattern, |v| >= 448 -> 448.
__device__ __forceinline__ uint32_t e4m3_rne_sat(float v) {
  const uint32_t u = __float_as_uint(v);
  const uint32_t sign = (u >> 24) & 0x80u;
  const uint32_t a = u & 0x7FFFFFFFu;
  if (a >= 0x43E00000u) return sign | 0x7Eu;           // >= 448
  const int e = (int)(a >> 23) - 127;
  uint32_t code;
  if (e >= -6) {                                        // normal result
    const uint32_t mant = a & 0x7FFFFFu;
    const uint32_t keep = mant >> 20, rem = mant & 0xFFFFFu;
    code = ((uint32_t)(e + 7) << 3) | keep;
    if (rem > 0x80000u || (rem == 0x80000u && (keep & 1u))) code += 1u;
  } else {                                              // subnormal: k * 2^-9
    const int shift = 14 - e;                           // >= 21
    if (shift > 24 || a < 0x00800000u) {
      code = 0u;                                        // < 2^-10 (or fp32 subnormal)
    } else {
      const uint32_t sig = (a & 0x7FFFFFu) | 0x800000u;
      const uint32_t keep = sig >> shift;
      const uint32_t rem = sig & ((1u << shift) - 1u);
      const uint32_t half = 1u << (shift - 1);
      code = keep + ((rem > half || (rem == half && (keep & 1u))) ? 1u : 0u);
    }
  }
  return sign | code;
}

__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  float v;
  if (e == 0) v = (float)m * 0.001953125f;                     // m * 2^-9
  else v = __uint_as_float(((e + 120u) << 23) | (m << 20));    // (1+m/8) 2^(e-7)
  return (c & 0x80u) ? -v : v;
}

// MX (OCP v1.0) block scale for E2M1: E = floor(log2 amax) - 2, clamped to
// [-127, 127]; returns E + 127 (0 when amax == 0).
__device__ __forceinline__ uint32_t e8m0_block_code(float amax) {
  const uint32_t u = __float_as_uint(amax) & 0x7FFFFFFFu;
  if (u == 0) return 0u;
  int fl;
  const uint32_t ef = u >> 23;
  if (ef != 0) fl = (int)ef - 127;
  else fl = (31 - __clz(u)) - 149;                              // fp32 subnormal
  int E = fl - 2;
  E = E < -127 ? -127 : (E > 127 ? 127 : E);
  return (uint32_t)(E + 127);
}

// 2^-(code-127) as fp32 (code in [0, 252] here, so it is a normal number).
__device__ __forceinline__ float e8m0_inv_scale(uint32_t code) {
  return __uint_as_float((254u - code) << 23);
}

// ---- generic helpers ----------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }
__device__ __forceinline__ int warp_id() { return threadIdx.x >> 5; }

// Time budget of every spin-wait, in SM clocks (about 1-2 s).
constexpr long long kWaitBudget = 3000000000LL;

// ---- mbarrier -------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Programmatic dependent launch.  pdl_wait: block until the previous kernel
// in the stream has completed and its writes are visible (a no-op when the
// kernel was launched without the attribute).  pdl_trigger: let the next
// kernel in the stream start its prologue now; it still waits for this
// kernel's completion before it reads what this kernel writes.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// The suspend-time hint lets a waiting thread sleep until the phase completes
// (or the hint, in ns, runs out) instead of spinning: spinning warps would take
// issue slots from the warps doing the work.
constexpr uint32_t kSuspendHintNs = 20000;
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}
// test_wait never suspends the thread, so a loop around it spins: for waits
// on the latency-critical path, where the waiter has nothing else to do and
// must resume as soon as the phase completes.
__device__ __forceinline__ bool mbar_try_wait_poll(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on a phase: false when `budget` SM clocks ran out first.
template <bool kPoll = false>
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, long long budget) {
  auto probe = [&] { return kPoll ? mbar_try_wait_poll(bar, parity) : mbar_try_wait(bar, parity); };
  if (probe()) return true;
  const long long t0 = clock64();
  while (!probe()) {
    if (clock64() - t0 > budget) return false;
  }
  return true;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait_for(bar, parity, kWaitBudget);
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Make generic-proxy shared-memory writes visible to the async proxy
// (tcgen05.mma / tcgen05.cp / TMA read shared memory through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- bulk copies ----------------------------------------------------------------
// Plain bulk copy global -> shared (16-B aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---- tcgen05 ----------------------------------------------------------------------------------
// Shared-memory matrix descriptor: start, leading-dimension byte offset,
// stride-dimension byte offset (all >> 4), descriptor version 1 (bit 46),
// swizzle mode in bits 61..63 (0 none, 2 = 128 B, 4 = 64 B, 6 = 32 B).
constexpr uint32_t kSwizzleNone = 0, kSwizzle128B = 2, kSwizzle64B = 4, kSwizzle32B = 6;
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swizzle << 61);
}

// Instruction descriptor, kind::f16 with fp16 A/B and fp32 accumulate.
// a_mn / b_mn: 1 when that operand is MN-major (else K-major).
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t M, uint32_t N, uint32_t a_mn, uint32_t b_mn) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) |
         ((M >> 4) << 24);
}
// Instruction descriptor, kind::mxf4 (E2M1 x E2M1, UE8M0 scales, K = 64).
// sfa_id / sfb_id select the byte of the 32-bit scale cell (0 or 2 for 2X).
__host__ __device__ constexpr uint32_t idesc_mxf4(uint32_t M, uint32_t N, uint32_t sfa_id, uint32_t sfb_id) {
  return (sfb_id << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24) |
         (sfa_id << 29);
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
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
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// Copy a 32-row x 16-byte shared-memory block into TMEM, replicated into all
// four 32-lane quarters (4 columns).
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 bit, 16 consecutive columns -> 16 registers per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// 32 lanes x 32 bit, 32 consecutive columns -> 32 registers per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
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
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}

}  // namespace csa
