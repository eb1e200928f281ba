// Device helpers for the tcgen05 (tensor memory) decode kernels: shared
// memory matrix descriptors, the f16 instruction descriptor, MMA issue and
// commit, bounded mbarrier waits, tensor-memory loads and stores, and the
// 128-byte-swizzled operand layout.
#pragma once

#include "decode_common.cuh"

namespace mlalb {
namespace tc {

constexpr long long kWaitCycles = 2000000000LL;  // ~1 s at 2 GHz

__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  // 128-byte swizzle, descriptor version 1
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ uint32_t idesc(int M, int N, int a_mn, int b_mn) {
  // f16 x f16 -> f32
  return (1u << 4) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, int acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"(acc));
}

__device__ __forceinline__ void commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void bar_init(uint32_t bar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void bar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One test of an mbarrier phase (no suspension).
__device__ __forceinline__ bool bar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase; on time-out raises the CTA abort flag.
// A phase that is already complete costs one test: the clock and the abort
// flag are read only when the thread has to wait (reading the clock behind
// outstanding tensor-core work costs a few hundred cycles).
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                         int32_t* err, long long limit = kWaitCycles) {
  if (bar_test(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (bar_test(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > limit) {
      *abort = 1;
      set_error(err, MLA_LOWBIT_DEV_PIPELINE);
      return false;
    }
  }
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float* v) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// 24 consecutive columns of this thread's lane as an x16 and an x8 load (in
// the order that keeps each naturally aligned: x8 first when the start is not
// a multiple of 16), one wait.
__device__ __forceinline__ void tmem_ld24(uint32_t taddr, float* v) {
  uint32_t r[24];
  const bool a16 = (taddr & 15u) == 0;
  const uint32_t t16 = a16 ? taddr : taddr + 8, t8 = a16 ? taddr + 16 : taddr;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(t16));
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                 "=r"(r[22]), "=r"(r[23])
               : "r"(t8));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  if (a16) {
#pragma unroll
    for (int i = 0; i < 24; ++i) v[i] = __uint_as_float(r[i]);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[16 + i]);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[8 + i] = __uint_as_float(r[i]);
  }
}

// cp.async of 4, 8 or 16 bytes (global -> shared), one commit group per tile
__device__ __forceinline__ void cp_async(void* dst, const void* src, int bytes) {
  const uint32_t d = su32(dst);
  if (bytes == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
  else if (bytes == 8)
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(d), "l"(src) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// byte offset of fp16 element e (0..63) of row r inside a 128-byte-swizzled block
__device__ __forceinline__ int sw_off(int r, int e) {
  return (r >> 3) * 1024 + (r & 7) * 128 + ((((e >> 3) ^ (r & 7))) << 4) + (e & 7) * 2;
}
// byte offset of 16-byte chunk c of row r
__device__ __forceinline__ int sw_chunk(int r, int c) {
  return (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4);
}

// Physical channel (0..63 in its group) held at position e of logical chunk c of
// a plane row, for the INT4 (type A) or INT2 (type B) unpack order.
__device__ __forceinline__ int chan_of_pos(int c, int e, bool typeB) {
  if (!typeB) return 8 * c + ((e & 1) ? 4 : 0) + (e >> 1);  // [0,4,1,5,2,6,3,7]
  const int base = 16 * (c >> 1) + ((c & 1) ? 4 : 0);       // [0,8,1,9,..] / [4,12,5,13,..]
  return base + ((e & 1) ? 8 : 0) + (e >> 1);
}

// ---------------------------------------------------------------- shared by the
// cluster kernels: A operand in tensor memory, tensor-memory stores and loads,
// cluster rank / barrier / peer addressing, st.async exchange, bounded waits

__device__ __forceinline__ void mma_tmem_a(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id,
                                           int acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(id), "r"(acc));
}

__device__ __forceinline__ void tmem_st16_nowait(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st8_nowait(uint32_t taddr, const uint32_t* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

__device__ __forceinline__ void tmem_st4_nowait(uint32_t taddr, const uint32_t* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3])
               : "memory");
}

// 12 consecutive columns as an x8 and an x4 store, each naturally aligned
// (the start is a multiple of 4).
__device__ __forceinline__ void tmem_st12_nowait(uint32_t taddr, const uint32_t* v) {
  if ((taddr & 7u) == 0) {
    tmem_st8_nowait(taddr, v);
    tmem_st4_nowait(taddr + 8, v + 8);
  } else {
    tmem_st4_nowait(taddr, v);
    tmem_st8_nowait(taddr + 4, v + 4);
  }
}

// 32 consecutive columns of this thread's lane, one wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  tmem_st16(taddr, v);
  tmem_st16(taddr + 16, v + 16);
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_peer(uint32_t addr, uint32_t peer) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(peer));
  return r;
}
// 16 bytes into the peer's shared memory, counted as transaction bytes on the
// peer's mbarrier (no fence: the barrier's phase completes once the bytes land).
__device__ __forceinline__ void st_async4(uint32_t addr, float a0, float a1, float a2, float a3,
                                          uint32_t bar_cluster_addr) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1,%2,%3,%4}, [%5];" ::"r"(addr),
      "f"(a0), "f"(a1), "f"(a2), "f"(a3), "r"(bar_cluster_addr)
      : "memory");
}
__device__ __forceinline__ void expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// Arrival on the peer's barrier that orders nothing: it only reports that this
// thread's reads of its buffer have returned.
__device__ __forceinline__ void arrive_peer_relaxed(uint32_t bar_cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster_addr)
               : "memory");
}
// Bounded wait for arrivals from the peer that carry no data.
__device__ __forceinline__ bool bar_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort,
                                                 int32_t* err, long long limit = kWaitCycles) {
  long long t0 = -1;
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.relaxed.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(200000u)
        : "memory");
    if (ok) return true;
    if (*abort) return false;
    if (t0 < 0) t0 = clock64();
    if (clock64() - t0 > limit) {
      *abort = 1;
      set_error(err, MLA_LOWBIT_DEV_PIPELINE);
      return false;
    }
  }
}
// Bounded wait on a local mbarrier phase; the thread sleeps in the barrier
// (up to kSuspendNs per try) instead of spinning, so waiting warps leave the
// issue slots to the working ones.
constexpr uint32_t kSuspendNs = 200000;
__device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, volatile int* abort, int32_t* err,
                                     long long limit = kWaitCycles) {
  if (bar_test(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
    if (ok) return true;
    if (*abort) return false;
    if (clock64() - t0 > limit) {
      *abort = 1;
      set_error(err, MLA_LOWBIT_DEV_PIPELINE);
      return false;
    }
  }
}

// x = hi + lo with hi = x cut to 11 significant bits (exact in fp16 over its
// normal range) and lo = the exact float32 remainder rounded to fp16: x to
// about 2^-21 relative, in fewer instructions than rounding hi.
__device__ __forceinline__ void split_trunc(float a, float b, uint32_t& hi, uint32_t& lo) {
  const float ha = __uint_as_float(__float_as_uint(a) & 0xFFFFE000u);
  const float hb = __uint_as_float(__float_as_uint(b) & 0xFFFFE000u);
  hi = pack_half2(ha, hb);
  lo = pack_half2(a - ha, b - hb);
}

// The same in bf16: hi = x cut to 8 significant bits (its upper 16 bits, exact
// in bf16), lo = the exact remainder rounded to bf16: x to about 2^-17
// relative, with fp32's exponent range.  Pairs are (a, b) in (low, high) halves.
__device__ __forceinline__ void split_trunc_bf16(float a, float b, uint32_t& hi, uint32_t& lo) {
  const uint32_t ua = __float_as_uint(a) & 0xFFFF0000u, ub = __float_as_uint(b) & 0xFFFF0000u;
  hi = ub | (ua >> 16);
  const float ra = a - __uint_as_float(ua), rb = b - __uint_as_float(ub);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(rb), "f"(ra));
}

}  // namespace tc
}  // namespace mlalb
