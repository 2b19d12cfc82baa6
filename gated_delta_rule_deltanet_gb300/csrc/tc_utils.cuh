// tc_utils.cuh -- thin inline-PTX wrappers for Blackwell (sm_103a) tensor cores:
// tensor memory (TMEM) allocation and access, tcgen05.mma with shared-memory
// and TMEM operands, completion through mbarriers, and the shared-memory matrix
// descriptor for the no-swizzle K-major "core matrix" layout.
//
// Operand layout used throughout (16-bit elements, K-major, no swizzle): a
// tile of R rows x K elements is a grid of core matrices, each 8 rows x 16
// bytes (8 elements) stored as 128 contiguous bytes (row r of the core matrix
// at byte 16 r).  Core matrices adjacent along K are `lbo` bytes apart, 8-row
// groups are `sbo` bytes apart.  One kind::f16 MMA consumes K = 16 (two core
// matrices along K), so successive K steps advance the start address by 2*lbo.
#pragma once

#include <stdint.h>

namespace kda {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of element (row, k) of a 16-bit K-major core-matrix tile.
__host__ __device__ __forceinline__ uint32_t cm_offset(uint32_t row, uint32_t k, uint32_t lbo,
                                                        uint32_t sbo) {
  return (row >> 3) * sbo + (k >> 3) * lbo + (row & 7) * 16 + (k & 7) * 2;
}

// MN-major (transposed) operand tiles, no swizzle: a core matrix is 8 K-rows of 16 bytes
// (8 consecutive M or N elements each), 128 contiguous bytes; core matrices adjacent
// along K are `lbo` bytes apart and along M/N `sbo` bytes apart (the same roles of the two
// offsets as in the K-major layout).  Byte offset of element (k, mn):
__host__ __device__ __forceinline__ uint32_t mn_offset(uint32_t k, uint32_t mn, uint32_t lbo,
                                                        uint32_t sbo) {
  return (k >> 3) * lbo + (mn >> 3) * sbo + (k & 7) * 16 + (mn & 7) * 2;
}

// ------------------------------------------------------------------ descriptors

// Shared-memory matrix descriptor: start address, leading (K) and stride (8-row)
// byte offsets, descriptor version 1, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo & 0x3FFFFu) >> 4) << 16;
  d |= static_cast<uint64_t>((sbo & 0x3FFFFu) >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // version
  return d;                             // base offset 0, absolute-LBO off, layout 0 (no swizzle)
}

// Descriptor of a K-major operand in the 128-byte swizzled layout that a TMA copy with
// 128-byte swizzle writes: rows of 128 bytes, the eight 16-byte chunks of row r stored at
// chunk ^ (r % 8), 8-row atoms `sbo` bytes apart; the region must be 1024-byte aligned.
// A K step of 16 elements within the 128-byte row advances the start address by 32 bytes.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t sbo) {
  return smem_desc(saddr, 16, sbo) | (static_cast<uint64_t>(2) << 61);
}

// Byte offset of the 16-byte chunk holding elements [8 c8, 8 c8 + 8) of row r in that layout
// (rows of 128 bytes from a 1024-byte aligned base).
__host__ __device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t c8) {
  return r * 128 + ((c8 ^ (r & 7)) << 4);
}

// The same descriptor with its start address advanced by `bytes` (a multiple of 16 that
// keeps the address inside shared memory, so the 14-bit field cannot carry).
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

enum : uint32_t { kF16 = 0, kBF16 = 1, kTF32 = 2 };   // A/B type field (kind::f16 / kind::tf32)

// Instruction descriptor of kind::f16: fp32 accumulator, A/B element types, optional
// negation of A, operands K-major unless a_mn / b_mn (MN-major), shape M x N.
__host__ __device__ __forceinline__ uint32_t idesc_f16(uint32_t M, uint32_t N, uint32_t ab_type,
                                                        bool neg_a = false, bool a_mn = false,
                                                        bool b_mn = false) {
  return (1u << 4)                      // D = f32
         | (ab_type << 7) | (ab_type << 10)
         | (neg_a ? (1u << 13) : 0u)
         | (a_mn ? (1u << 15) : 0u) | (b_mn ? (1u << 16) : 0u)
         | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete, giving up after
// `limit` polls; returns false on timeout (the caller records an error).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One arrival that also announces `bytes` of asynchronous copies completing on `bar`.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Barrier `id` (1..15) among the first `count` threads that reach it (a multiple of 32).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Barrier `id` among the first `count` threads that reach it, returning whether `pred`
// held in any of them, so that every participant takes the same branch afterwards.
__device__ __forceinline__ bool named_sync_or(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// ------------------------------------------------------------------ fences

// Makes generic-proxy shared-memory writes visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------------ TMEM

// Executed by one full warp.  `dst` receives the TMEM base address.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: thread t of the warp receives
// columns [col, col+16) of lane (lane_base + t).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
// 32 lanes x 8 consecutive 32-bit columns (thread t writes lane lane_base + t).
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ MMA

// D[tmem] (+)= A[smem] * B[smem]^T, one instruction (K = 16 for kind::f16).
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same with A read from tensor memory (row i = lane i, two 16-bit elements per column).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// kind::tf32: A and B are fp32 in shared memory, read with a 10-bit mantissa (K = 8 per
// instruction: 32 bytes of a K-major row, the same byte step as kind::f16's K = 16).
__device__ __forceinline__ void mma_ss_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on `bar` when every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------------ async copies

// 16-byte global -> shared copy that bypasses registers; bytes beyond
// `src_bytes` (0 or 16) are zero-filled.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}
// Waits until at most one committed group of this thread is still in flight.
__device__ __forceinline__ void cp_async_wait_one() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// Bulk (TMA-engine) copy of `bytes` (multiple of 16, both addresses 16-byte aligned)
// from global to shared memory; completion is counted in bytes on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t sdst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          sdst),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// L2 prefetch of one box of a tiled tensor map: no shared memory and no barrier involved
__device__ __forceinline__ void tma_prefetch_3d(const void* map, int32_t x, int32_t y, int32_t z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(map), "r"(x),
               "r"(y), "r"(z)
               : "memory");
}

// Tiled 2-D TMA load of one box of `map` at element coordinates (x, y) into shared memory;
// completion is counted in bytes on `bar`.  x * element size must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(uint32_t sdst, const void* map, int32_t x, int32_t y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(sdst),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Tiled 3-D TMA load of one box of `map` at element coordinates (x, y, z) into shared
// memory; completion is counted in bytes on `bar`.  x * element size must be a multiple of 16.
__device__ __forceinline__ void tma_load_3d(uint32_t sdst, const void* map, int32_t x, int32_t y,
                                            int32_t z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(sdst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// Bulk (TMA-engine) copy of `bytes` (multiple of 16, both addresses 16-byte aligned)
// from shared to global memory, tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_store(void* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(ssrc), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until every committed bulk group of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ------------------------------------------------------------------ conversions

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ------------------------------------------------------------------ operand tiles

// dense K-major tiles: lbo 128, sbo = (K / 8) * 128
__host__ __device__ constexpr uint32_t dense_sbo(uint32_t K) { return (K / 8) * 128; }

// 8 fp32 values -> 8 fp16 (round to nearest even) at a 16-byte aligned offset
__device__ __forceinline__ void f16x8_store(unsigned char* smem, uint32_t off, const float* x) {
  uint4 v;
  v.x = pack_f16x2(x[0], x[1]);
  v.y = pack_f16x2(x[2], x[3]);
  v.z = pack_f16x2(x[4], x[5]);
  v.w = pack_f16x2(x[6], x[7]);
  *reinterpret_cast<uint4*>(smem + off) = v;
}

__device__ __forceinline__ uint16_t f16_bits(float x) {
  return static_cast<uint16_t>(pack_f16x2(x, 0.f) & 0xffffu);
}

// element idx of a bf16 array at byte offset `off`, widened exactly to fp32
__device__ __forceinline__ float bf16_at(const unsigned char* smem, uint32_t off, int idx) {
  return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(smem + off)[idx])
                         << 16);
}

// 8 bf16 from a 16-byte aligned address, widened to fp32
__device__ __forceinline__ void bf16x8_load(const unsigned char* p, float* x) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    x[2 * e] = __uint_as_float(w[e] << 16);
    x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
  }
}

// 8 fp16 from a 16-byte aligned address, widened to fp32
__device__ __forceinline__ void f16x8_load(const unsigned char* p, float* x) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e)
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
        : "=f"(x[2 * e]), "=f"(x[2 * e + 1]) : "r"(w[e]));
}

}  // namespace tc
}  // namespace kda
