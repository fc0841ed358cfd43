// Device helpers shared by the flint_moe kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#define FLINT_DEV __device__ __forceinline__

namespace flint {

// ------------------------------------------------------------------ bf16 --
FLINT_DEV float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// fp32 -> bf16 bits, round to nearest even (cvt.rn.bf16.f32).
FLINT_DEV uint32_t f32_to_bf16_bits(float f) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}

FLINT_DEV float round_bf16(float f) { return __bfloat162float(__float2bfloat16_rn(f)); }

// ------------------------------------------------------------------ NVFP4 --
// Two e2m1 codes -> one bf16x2 holding e2m1(code) * 2^-126 each, exactly.
// Placing the code's exponent/mantissa bits (c = bits 2..0) at bf16 bits 8..6
// makes the bf16 exponent field equal to the e2m1 exponent field, so the
// bf16 value is 2^(E-127) * (1 + m/2) = e2m1 * 2^-126 for E > 0 and the bf16
// subnormal m/2 * 2^-126 = e2m1 * 2^-126 for E = 0; the sign goes to bit 15.
// `v` carries code A in bits 3..0 and code B in bits 19..16.
// Both moves are one multiply: a 4-bit field times 2^6 + 2^12 lands at bits
// 6..9 and 12..15 without overlap (so without carries), and the mask keeps
// bits 6..8 of the first copy and bit 15 (the sign) of the second.
FLINT_DEV uint32_t e2m1x2_to_bf16x2_scaled(uint32_t v) {
  return ((v & 0x000F000Fu) * 0x1040u) & 0x81C081C0u;
}

// Pair `a` (0..3) of a word of 8 codes (nibble i = K offset i): codes a and
// a + 4 as (lo, hi) of a bf16x2, each e2m1 * 2^-126.
FLINT_DEV uint32_t e2m1_pair(uint32_t word, int a) {
  return e2m1x2_to_bf16x2_scaled(word >> (4 * a));
}

// Two e4m3 block-scale bytes (lo = bits 7..0, hi = bits 15..8 of `b2`) ->
// bf16x2 of scale * 2^119 each, exact: e4m3 -> f16 is exact (hardware cvt),
// the fp32 product with 2^119 is exact (max 448 * 2^119 < 2^128) and the
// result has at most 4 significant bits, so the bf16 rounding is exact.
FLINT_DEV uint32_t e4m3x2_to_bf16x2_x2p119(uint32_t b2) {
  uint32_t h2;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h2) : "r"(b2));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  const float k = __int_as_float((119 + 127) << 23);  // 2^119
  float lo = __low2float(h) * k;
  float hi = __high2float(h) * k;
  __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&r);
}

FLINT_DEV uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hmul2(*reinterpret_cast<__nv_bfloat162*>(&a),
                             *reinterpret_cast<__nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Broadcast the lo (sel 0) or hi (sel 1) bf16 of a bf16x2 to both halves.
FLINT_DEV uint32_t bf16x2_bcast(uint32_t v, int hi) {
  return hi ? __byte_perm(v, 0, 0x3232) : __byte_perm(v, 0, 0x1010);
}

// ------------------------------------------------------------ NVFP4 (f16) --
// The four code bytes of a word -> four f16x2 (byte b: low nibble = K 2b in
// the low half, high nibble = K 2b + 1 in the high half), by the hardware
// e2m1 -> f16 conversion (every e2m1 value is exact in f16).
FLINT_DEV void e2m1x8_to_f16x2(uint32_t word, uint32_t (&p)[4]) {
  asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0; cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2; cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(p[0]), "=r"(p[1]), "=r"(p[2]), "=r"(p[3])
      : "r"(word));
}
// Two e4m3 block-scale bytes -> f16x2 (exact: e4m3 values are f16 values).
FLINT_DEV uint32_t e4m3x2_to_f16x2(uint32_t b2) {
  uint32_t h2;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h2) : "r"(b2));
  return h2;
}
FLINT_DEV uint32_t f16x2_bcast(uint32_t v, int hi) {
  return hi ? __byte_perm(v, 0, 0x3232) : __byte_perm(v, 0, 0x1010);
}
// f16x2 product; exact for e2m1 x e4m3 (at most 6 significant bits, within
// f16's normal range).
FLINT_DEV uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// 2^e as fp32 for -126 <= e <= 127, by its bit pattern.
FLINT_DEV float pow2f(int e) { return __int_as_float((e + 127) << 23); }

// ------------------------------------------------------------ tensor core --
// D = A * B + D, m16n8k16, bf16 inputs, fp32 accumulators (mma.sync).
FLINT_DEV void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Same with f16 operands.
FLINT_DEV void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                             uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// --------------------------------------------------------------- memory --
FLINT_DEV uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

FLINT_DEV uint32_t ldg_nc_u16(const void* p) {
  unsigned short r;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
  return r;
}

// L2-coherent loads for data written by other CTAs of the same or an
// earlier, still-overlapping grid.
FLINT_DEV uint4 ldg_cg_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
FLINT_DEV int ldg_cg_i32(const int* p) {
  int r;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}
FLINT_DEV float ldg_cg_f32(const float* p) {
  float r;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(r) : "l"(p));
  return r;
}
FLINT_DEV uint32_t ldg_cg_u16(const void* p) {
  unsigned short r;
  asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(r) : "l"(p));
  return r;
}

// ------------------------------------------------ programmatic launches --
// Wait until the preceding grid in the stream has completed and its writes
// are visible (no-op when launched without the PDL attribute).
FLINT_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next grid in the stream to start launching.
FLINT_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// --------------------------------------------------------------- math --
// sigmoid as rcp.approx(1 + ex2.approx(-g * log2 e)); silu(g) = g * sigmoid(g).
FLINT_DEV float silu_approx(float g) {
  float e, r;
  asm("ex2.approx.f32 %0, %1;" : "=f"(e) : "f"(-g * 1.4426950408889634f));
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return g * r;
}

FLINT_DEV uint32_t ordered_bf16(uint32_t b) { return (b & 0x8000u) ? (b ^ 0xFFFFu) : (b | 0x8000u); }

}  // namespace flint

namespace flint {
// ------------------------------------------------ mbarrier / bulk copies --
FLINT_DEV uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
FLINT_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
FLINT_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
FLINT_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
// Adds `bytes` to the expected transaction count without arriving.
FLINT_DEV void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
FLINT_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Test for phase completion; if not complete the thread may be suspended
// (woken by the completion) for up to `hint_ns` before returning false.
// Non-blocking probe of the phase with the given parity.
FLINT_DEV bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
FLINT_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity, uint32_t hint_ns = 0) {
  uint32_t ok;
  if (hint_ns) {
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
  } else {
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
  }
  return ok != 0;
}
// 1-D bulk copy global -> shared, completion counted on `bar` (bytes).
FLINT_DEV void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// Named barrier among `nthreads` threads (multiple of 32).
FLINT_DEV void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
FLINT_DEV int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
FLINT_DEV void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
}  // namespace flint

namespace flint {
// Add without a returned value, release semantics (GPU scope).
FLINT_DEV void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Per-thread asynchronous 4-byte global -> shared copy (both addresses 4-byte
// aligned), tracked in the thread's copy groups.
FLINT_DEV void cp_async4(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(smem_dst)), "l"(gsrc)
               : "memory");
}
FLINT_DEV void cp_async8(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(smem_dst)), "l"(gsrc)
               : "memory");
}
FLINT_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's most recent copy groups are pending.
template <int N>
FLINT_DEV void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
FLINT_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

FLINT_DEV unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
}  // namespace flint

namespace flint {
// Shared-memory add with acquire-release semantics at CTA scope; returns old.
FLINT_DEV int atom_add_acqrel_cta_smem(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(smem_addr(p)), "r"(v)
               : "memory");
  return old;
}
// Order this thread's earlier generic-proxy global accesses (and what it has
// observed) before its later async-proxy (bulk copy) accesses.
FLINT_DEV void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// ------------------------------------------------------------------ spans --
// Kernel spans (flint_moe_record_spans): per kernel id and CTA (mod
// kSpanCtas) the CTA's start, stored as its bitwise complement so that
// atomicMax keeps the earliest, and the exit of its last warp.  The buffer
// address is a device variable of each translation unit (set by its
// span_buffer_set_*), read afresh at a CTA's start and at each warp's exit,
// so a guard holds no register through the kernel; its destructor runs on
// every return path, and with a null buffer it does nothing.
constexpr int kSpanCtas = 1024;
enum {
  kSpanRoute = 0, kSpanGateUp = 1, kSpanDown = 2, kSpanSingle = 3, kSpanGroupCount = 4,
  kSpanGroupScan = 5, kSpanGroupScatter = 6, kSpanPlan = 7, kSpanGather = 8, kSpanGemm1 = 9,
  kSpanGemm2 = 10, kSpanCombine = 11, kSpanAddNorm = 12, kSpanSharedGateUp = 13, kSpanSharedDown = 14,
  kSpanSharedAdd = 15, kSpanQkvGemv = 16, kSpanQkvHeads = 17
};
static __device__ unsigned long long* g_span_buf;
FLINT_DEV unsigned long long* span_slot(int id) {
  unsigned long long* b = *reinterpret_cast<unsigned long long* volatile*>(&g_span_buf);
  if (!b) return nullptr;
  return b + ((size_t)id * kSpanCtas + (blockIdx.x + gridDim.x * blockIdx.y) % kSpanCtas) * 2;
}
template <int ID>
struct SpanGuard {
  __device__ __forceinline__ SpanGuard() {
    if (threadIdx.x == 0) {
      unsigned long long* s = span_slot(ID);
      if (s) atomicMax(s, ~globaltimer_ns());
    }
  }
  __device__ __forceinline__ ~SpanGuard() {
    if ((threadIdx.x & 31) == 0) {
      unsigned long long* s = span_slot(ID);
      if (s) atomicMax(s + 1, globaltimer_ns());
    }
  }
};
// The host-side setter of this translation unit's buffer address.
#define FLINT_SPAN_SETTER(unit)                                        \
  cudaError_t span_buffer_set_##unit(unsigned long long* b) {          \
    return cudaMemcpyToSymbol(g_span_buf, &b, sizeof(b));              \
  }
// Generic-proxy shared-memory accesses ordered with the async proxy's (bulk
// copies and the tensor core read and write shared memory through it).
FLINT_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
}  // namespace flint
