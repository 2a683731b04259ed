// ptx.cuh -- thin inline-PTX wrappers for the sm_103a features the kernels
// use: mbarriers, TMA tensor loads, tcgen05 MMA / TMEM allocation, and the
// descriptors that tcgen05.mma reads.  Written from the public PTX ISA
// description of these instructions.
#pragma once
#include <cstdint>

namespace cpattn {

// ----------------------------------------------------------------- basics
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// 2^x on the SFU (approximate, flush-to-zero): the hot-loop exponential.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// fp32 bits -> the nearest tf32 (10 explicit mantissa bits), ties away
// from zero: half of the dropped range added to the magnitude bits carries
// into the kept bits exactly when the dropped part is at least half an ulp
// (into the exponent when the mantissa overflows), then the 13 dropped bits
// are cleared, so a kind::tf32 MMA reads the value exactly.  Two integer
// operations: the conversion instruction added three times as much time to
// the fp32 path.  NaNs whose payload lies only in the dropped bits become
// infinities, as under truncation.
__device__ __forceinline__ uint32_t tf32_round_bits(uint32_t x) {
  return (x + 0x1000u) & 0xFFFFE000u;
}

// max of three floats in one instruction (sm_100+).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Packed two-lane fp32 arithmetic (sm_100+): one instruction for two lanes.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                      float c0, float c1) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void fadd2(float& d0, float& d1, float a0, float a1, float b0,
                                      float b1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// One lane of the (fully active) warp, chosen by elect.sync: a leader the
// compiler treats as a uniform choice.
__device__ __forceinline__ bool elect_one() {
  uint32_t elected;
  asm volatile("{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}"
               : "=r"(elected));
  return elected != 0;
}

// Per-warpgroup register budget changes (all warps of a warpgroup execute
// the same one).  The block's launch allocation must cover the new split.
template <int N>
__device__ __forceinline__ void regs_increase() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_decrease() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Non-blocking check whether the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity.  Returns false when
// `timeout_ns` passes (then it raises the CTA's abort flag and ORs `code`
// into the device error word `err`), or when another thread of the CTA has
// already raised the abort flag.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          volatile int* abort_flag, uint64_t timeout_ns,
                                          unsigned int* err, unsigned code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > timeout_ns) {
      *abort_flag = 1;
      atomicOr(err, code);
      return false;
    }
  }
}

// Bounded wait that ignores the abort flag: used only to drain copies and
// MMAs that are already in flight before a CTA leaves after an abort.
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  return true;
}

// ----------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 4-D tiled tensor load global -> shared, completion counted on `bar` in
// bytes.  c0 is the innermost coordinate (elements).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap, uint32_t bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// L2 eviction policies for cache-hinted accesses: data read once (query
// tiles) or written once and not read again by the kernel (the final
// output) is marked evict-first, data that other CTAs read again (key and
// value tiles) evict-last, so the reused data is what stays in L2.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// tma_load_4d with an L2 cache policy.
__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const void* tmap, uint32_t bar,
                                                 int c0, int c1, int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "l"(policy)
      : "memory");
}

// 16-byte global store with an L2 cache policy.
__device__ __forceinline__ void st_global_v4_hint(void* ptr, uint4 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(ptr), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(policy)
               : "memory");
}

// 4-D tiled tensor prefetch into L2 (no shared-memory destination, no
// completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_4d(const void* tmap, int c0, int c1, int c2,
                                                   int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

// ----------------------------------------------------------------- tcgen05
// Orders this thread's earlier generic-proxy global accesses before later
// async-proxy (bulk copy) accesses that synchronise with it.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Untiled bulk copy global -> shared: both addresses 16-byte aligned, size a
// multiple of 16; the barrier's transaction count drops by `bytes` on arrival.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Whole warp: allocate `ncols` TMEM columns; the base address lands in smem.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T-ish per the instruction descriptor.
// kind::f16 covers bf16 operands, kind::tf32 fp32 (tf32) operands.
template <bool TF32>
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  if constexpr (TF32) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// Same with the A operand read from Tensor Memory.
template <bool TF32>
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  if constexpr (TF32) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// N bf16 MMAs (kind::f16) from one asm statement: D (+)= A_i B_i, the first
// accumulating into D iff acc != 0, the others always.  Operands are given
// as the low 32-bit words of their shared-memory descriptors with one shared
// high word (all descriptors here have equal strides, version and swizzle).
// SS: A is a shared-memory descriptor; TS: A is a TMEM address.  One
// statement keeps the issuing warp's instruction count per MMA minimal: that
// warp shares its SM sub-partition with busy softmax warps and gets few
// issue slots.
template <int N, bool SS>
__device__ __forceinline__ void mma_group(uint32_t d, const uint32_t* a, const uint32_t* b,
                                          uint32_t hi, uint32_t idesc, uint32_t acc);
template <>
__device__ __forceinline__ void mma_group<4, true>(uint32_t d, const uint32_t* a, const uint32_t* b,
                                                uint32_t hi, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t.reg .b64 ra, rb;\n\t"
      "setp.ne.b32 p, %10, 0;\n\tsetp.eq.b32 t, %10, %10;\n\t"
      "mov.b64 ra, {%1, %9};\n\t"
      "mov.b64 rb, {%5, %9};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %11, p;\n\t"
      "mov.b64 ra, {%2, %9};\n\t"
      "mov.b64 rb, {%6, %9};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %11, t;\n\t"
      "mov.b64 ra, {%3, %9};\n\t"
      "mov.b64 rb, {%7, %9};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %11, t;\n\t"
      "mov.b64 ra, {%4, %9};\n\t"
      "mov.b64 rb, {%8, %9};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %11, t;\n\t"
      "}\n" ::"r"(d), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]), "r"(b[2]), "r"(b[3]), "r"(hi), "r"(acc), "r"(idesc)
      : "memory");
}
template <>
__device__ __forceinline__ void mma_group<4, false>(uint32_t d, const uint32_t* a, const uint32_t* b,
                                                uint32_t hi, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t.reg .b64 ra, rb;\n\t"
      "setp.ne.b32 p, %10, 0;\n\tsetp.eq.b32 t, %10, %10;\n\t"
      "mov.b64 rb, {%5, %9};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], rb, %11, p;\n\t"
      "mov.b64 rb, {%6, %9};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], rb, %11, t;\n\t"
      "mov.b64 rb, {%7, %9};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], rb, %11, t;\n\t"
      "mov.b64 rb, {%8, %9};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], rb, %11, t;\n\t"
      "}\n" ::"r"(d), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]), "r"(b[2]), "r"(b[3]), "r"(hi), "r"(acc), "r"(idesc)
      : "memory");
}
template <>
__device__ __forceinline__ void mma_group<8, true>(uint32_t d, const uint32_t* a, const uint32_t* b,
                                                uint32_t hi, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t.reg .b64 ra, rb;\n\t"
      "setp.ne.b32 p, %18, 0;\n\tsetp.eq.b32 t, %18, %18;\n\t"
      "mov.b64 ra, {%1, %17};\n\t"
      "mov.b64 rb, {%9, %17};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %19, p;\n\t"
      "mov.b64 ra, {%2, %17};\n\t"
      "mov.b64 rb, {%10, %17};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %19, t;\n\t"
      "mov.b64 ra, {%3, %17};\n\t"
      "mov.b64 rb, {%11, %17};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %19, t;\n\t"
      "mov.b64 ra, {%4, %17};\n\t"
      "mov.b64 rb, {%12, %17};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %19, t;\n\t"
      "mov.b64 ra, {%5, %17};\n\t"
      "mov.b64 rb, {%13, %17};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %19, t;\n\t"
      "mov.b64 ra, {%6, %17};\n\t"
      "mov.b64 rb, {%14, %17};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %19, t;\n\t"
      "mov.b64 ra, {%7, %17};\n\t"
      "mov.b64 rb, {%15, %17};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %19, t;\n\t"
      "mov.b64 ra, {%8, %17};\n\t"
      "mov.b64 rb, {%16, %17};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %19, t;\n\t"
      "}\n" ::"r"(d), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]), "r"(b[0]), "r"(b[1]), "r"(b[2]), "r"(b[3]), "r"(b[4]), "r"(b[5]), "r"(b[6]), "r"(b[7]), "r"(hi), "r"(acc), "r"(idesc)
      : "memory");
}
template <>
__device__ __forceinline__ void mma_group<8, false>(uint32_t d, const uint32_t* a, const uint32_t* b,
                                                uint32_t hi, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t.reg .b64 ra, rb;\n\t"
      "setp.ne.b32 p, %18, 0;\n\tsetp.eq.b32 t, %18, %18;\n\t"
      "mov.b64 rb, {%9, %17};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], rb, %19, p;\n\t"
      "mov.b64 rb, {%10, %17};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], rb, %19, t;\n\t"
      "mov.b64 rb, {%11, %17};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], rb, %19, t;\n\t"
      "mov.b64 rb, {%12, %17};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], rb, %19, t;\n\t"
      "mov.b64 rb, {%13, %17};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], rb, %19, t;\n\t"
      "mov.b64 rb, {%14, %17};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%6], rb, %19, t;\n\t"
      "mov.b64 rb, {%15, %17};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], rb, %19, t;\n\t"
      "mov.b64 rb, {%16, %17};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%8], rb, %19, t;\n\t"
      "}\n" ::"r"(d), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]), "r"(b[0]), "r"(b[1]), "r"(b[2]), "r"(b[3]), "r"(b[4]), "r"(b[5]), "r"(b[6]), "r"(b[7]), "r"(hi), "r"(acc), "r"(idesc)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// Shared-memory matrix descriptor for a tile stored in the 128-byte swizzled
// canonical layout (rows of 128 bytes, 8-row / 1024-byte swizzle atoms).
//   lbo: byte distance between swizzle atoms along the leading (MN) dimension
//        of an MN-major operand; unused (encoded 1) for K-major.
//   sbo: byte distance between consecutive 8-row groups.
// Bits 46-47 hold the descriptor version (1), bits 61-63 the swizzle mode
// (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// Instruction descriptor for kind::f16 / kind::tf32 with fp32 accumulation.
//   ab_format: 1 = bf16, 2 = tf32.  b_mn_major: B stored MN-major.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t ab_format, bool b_mn_major, int m, int n) {
  return (1u << 4)                                  // D format: f32
         | (ab_format << 7) | (ab_format << 10)     // A, B formats
         | (static_cast<uint32_t>(b_mn_major) << 16)
         | (static_cast<uint32_t>(n >> 3) << 17)
         | (static_cast<uint32_t>(m >> 4) << 24);
}

}  // namespace cpattn
