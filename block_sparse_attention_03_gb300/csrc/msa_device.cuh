// Device-side building blocks shared by the MSA kernels (sm_103a).
//
// - mbarrier + bulk / tensor (TMA) copies into shared memory, with every wait
//   bounded: a wait that gives up sets MSA_FLAG_TIMEOUT in the status word and
//   the caller skips the work instead of hanging;
// - warp-level tensor-core MMA wrappers (mma.sync e4m3 k32 / bf16 k16 / f16 k16);
// - small conversions (fp32 pairs -> packed e4m3 / bf16 / f16).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace msa {

constexpr int kBlock = 128;  // tokens per paged block
constexpr int kDim = 128;    // head_dim == index_dim

// status word bits (sticky, first word of the workspace)
constexpr uint32_t FLAG_BAD_BLOCK = 1u << 0;    // block-table entry outside the pool
constexpr uint32_t FLAG_BAD_SEQLEN = 1u << 1;   // seq_len outside [q_per_seq, max_blocks*128]
constexpr uint32_t FLAG_BAD_SELECT = 1u << 2;   // selected block the query cannot see
constexpr uint32_t FLAG_TIMEOUT = 1u << 3;      // a bounded wait gave up

struct DeviceStatus {
  uint32_t flags;
  int32_t detail;
};

__device__ __forceinline__ void raise_flag(DeviceStatus* st, uint32_t f, int32_t detail) {
  if (st != nullptr) {
    atomicOr(&st->flags, f);
    atomicExch(&st->detail, detail);
  }
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Plain arrival (no transaction bytes): completes a phase whose only
// expected arrival is this one.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Wait until the phase with the given parity completes.  Bounded: each
// try_wait returns after a short, implementation-defined time if the phase is
// still open; after ~max_tries of them (a few seconds at most) it gives up and
// returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int max_tries = 4000000) {
  const uint32_t a = smem_u32(bar);
#pragma unroll 1
  for (int i = 0; i < max_tries; ++i) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// The same wait for kernels whose warps wait long and many at a time (the
// prefill indexer and attend): each try_wait may suspend the thread for up to
// kWaitSuspendNs, woken by the phase's completion, instead of re-testing
// (the re-tests of many waiting warps kept the shared-memory pipe busy);
// max_tries of them take at most max_tries x 10 us (2 s by default).  The
// decode kernels' short, latency-critical waits keep the plain test.
constexpr uint32_t kWaitSuspendNs = 10000;
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, int max_tries = 200000) {
  const uint32_t a = smem_u32(bar);
#pragma unroll 1
  for (int i = 0; i < max_tries; ++i) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(a), "r"(parity), "n"(kWaitSuspendNs)
        : "memory");
    if (done) return true;
  }
  return false;
}

// Warp-uniform wait: every lane polls, the warp agrees on the outcome.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, int max_tries = 4000000) {
  const uint32_t a = smem_u32(bar);
#pragma unroll 1
  for (int i = 0; i < max_tries; ++i) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (__all_sync(0xffffffffu, done)) return true;
  }
  return false;
}

// Order this thread's earlier generic-proxy accesses to shared memory before
// later async-proxy (bulk / tensor copy) writes to it.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 1-D bulk copy global -> shared; both addresses 16-B aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 1-D bulk copy shared -> global, tracked by this thread's bulk groups; both
// addresses 16-B aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Until this thread's committed bulk copies have read their shared-memory sources.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Until they have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// 2-D tensor (TMA) copy global -> shared at element coordinates (x, y).
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int32_t x, int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// The same copies with an L2 cache policy (createpolicy) for the source lines.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const void* tmap, int32_t x, int32_t y, uint64_t* bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// Policy for data read once as a stream: its lines are the first L2 evicts,
// so that what the next kernels read (block tables, scores, their code) stays.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ---------------------------------------------------------------- named barriers (ids > 0)

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Barrier over nthreads threads that also returns the OR of their predicates.
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 q, %1, 0; bar.red.or.pred p, %2, %3, q; selp.u32 %0, 1, 0, p; }"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// ---------------------------------------------------------------- PDL

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// ---------------------------------------------------------------- MMA (warp-level)

// D[16x8] += A[16x32] * B[32x8], e4m3 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_e4m3_k32(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D[16x8] += A[16x16] * B[16x8], bf16 inputs.
__device__ __forceinline__ void mma_bf16_k16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D[16x8] += A[16x16] * B[16x8], f16 inputs.
__device__ __forceinline__ void mma_f16_k16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four 8x8 b16 matrices from shared memory (row addresses from lanes 0-31).
__device__ __forceinline__ void ldmatrix_x4(uint32_t r[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t r[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// ---------------------------------------------------------------- conversions

// Pack two floats into e4m3x2 (lo -> byte 0), round to nearest even, saturating.
__device__ __forceinline__ uint16_t pack_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("{ .reg .b16 t; cvt.rn.satfinite.e4m3x2.f32 t, %1, %2; mov.b16 %0, t; }" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Decode two e4m3 bytes (byte 0 -> .x) to floats exactly.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v) {
  uint32_t h;
  asm("{ .reg .b16 t; mov.b16 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h) : "h"(v));
  __half2 hh = *reinterpret_cast<__half2*>(&h);
  return __half22float2(hh);
}

// Decode one e4m3 byte exactly.
__device__ __forceinline__ float e4m3_to_float(uint8_t v) { return e4m3x2_to_float2(v).x; }

// Decode two e2m1 nibbles of one byte (low nibble -> .x) to f16x2 exactly.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t h;
  asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h) : "r"(byte));
  return h;
}

// Two f16 values rounded to E4M3 (nearest, ties to even, saturating at
// +-448) and widened back to f16 exactly.
__device__ __forceinline__ uint32_t e4m3_round_f16x2(uint32_t h) {
  uint32_t r;
  asm("{ .reg .b16 t; cvt.rn.satfinite.e4m3x2.f16x2 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(r) : "r"(h));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Split x (|x| <= 448) into e4m3 hi + lo with x ~= hi + lo to ~8 significant bits.
__device__ __forceinline__ void split_e4m3(float x, float& hi, float& lo) {
  uint16_t h = pack_e4m3x2(x, 0.f);
  hi = e4m3x2_to_float2(h).x;
  lo = x - hi;
}

// Largest e with amax * 2^e <= lim (amax > 0 and finite); 0 for zero, NaN or
// infinite amax.  The corrections after the frexp estimate are bounded, so
// any input ends.
__device__ __forceinline__ int pow2_fit(float amax, float lim) {
  if (!(amax > 0.f) || !(amax <= 3.0e38f)) return 0;
  int e;
  frexpf(lim / amax, &e);  // lim/amax = f * 2^e, f in [0.5, 1)
  e -= 1;
  for (int t = 0; t < 4 && ldexpf(amax, e) > lim; ++t) --e;
  for (int t = 0; t < 4 && ldexpf(amax, e + 1) <= lim; ++t) ++e;
  return e;
}

// 2^e as a float for e in [-126, 127].
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }

// Largest e with v * 2^e <= 448 for a normal v > 0 (448 = 1.75 * 2^8), from
// the exponent and mantissa fields; other v go the general way.
__device__ __forceinline__ int fit448(float v) {
  const uint32_t u = __float_as_uint(v);
  const int be = (int)((u >> 23) & 0xffu);
  if (!(v > 0.f) || be == 0 || be == 255) return pow2_fit(v, 448.f);
  const int E = be - 127;
  return ((u & 0x7fffffu) <= 0x600000u ? 8 : 7) - E;
}

// Order-preserving map of a float to uint32 (NaN sorts as -inf - 1; -0 and +0
// map to one key, as they compare equal).
__device__ __forceinline__ uint32_t float_order_key(float f) {
  if (f != f) return 0u;
  uint32_t u = __float_as_uint(f);
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float order_key_float(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

}  // namespace msa
