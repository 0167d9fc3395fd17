// tc_common.cuh -- sm_103a building blocks for the tensor-core kernels:
// mbarriers with bounded waits, TMA tile copies, tcgen05 (TMEM allocation,
// MMA issue/commit, TMEM loads) and the shared-memory operand layouts.
//
// Operand layouts (bf16, 128-byte swizzle).  A tile is stored as rows of 64
// elements (128 B); 8 consecutive rows form a 1024-B swizzle atom in which
// the 16-B chunk c of row r sits at chunk position c ^ (r % 8).  A logical
// [R rows][X cols] tile with X a multiple of 64 is kept as X/64 column blocks
// of R rows each, block b at byte b * R * 128:
//     offset(r, x) = (x/64)*R*128 + (r/8)*1024 + (r%8)*128
//                    + ((((x%64)/8) ^ (r%8)) * 16) + (x%8)*2
// The same bytes serve two MMA roles:
//   K-major operand  (rows = M or N index, x = K index): SBO = 1024 between
//     8-row groups; a 16-wide K step starts 32 B further inside the atom,
//     K blocks of 64 are R*128 B apart;
//   MN-major operand (rows = K index, x = M or N index): SBO = 1024 between
//     8-row K groups, LBO = R*128 between 64-wide MN blocks; a 16-row K step
//     starts 2048 B further.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace slim {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- layouts --------------------------------------------------------------

__host__ __device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t x, uint32_t rows) {
  return (x >> 6) * rows * 128u + (r >> 3) * 1024u + (r & 7u) * 128u +
         ((((x & 63u) >> 3) ^ (r & 7u)) << 4) + (x & 7u) * 2u;
}

// tcgen05 shared-memory matrix descriptor.
//   bits  0-13 start address >> 4      bits 16-29 leading byte offset >> 4
//   bits 32-45 stride byte offset >> 4 bits 46-47 version (1)
//   bits 49-51 base offset (0: atoms are 1024-B aligned)
//   bits 61-63 swizzle: 0 none, 2 = 128 B
__device__ __forceinline__ uint64_t make_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(swizzle & 7u) << 61;
  return d;
}

constexpr uint32_t kSwizzle128 = 2;

// The start address is the low field of a descriptor, in 16-byte units, and
// no operand crosses the 256 KB it can address, so stepping along K is an
// integer add to a loop-invariant base descriptor.

// K-major operand: rows [row0, row0 + extent) of a `rows`-row tile, K step s
// (16 elements).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, uint32_t rows, uint32_t row0,
                                                uint32_t s) {
  return make_desc(base + (row0 >> 3) * 1024u, 16u, 1024u, kSwizzle128) +
         (uint64_t)((s >> 2) * rows * 8u + (s & 3u) * 2u);
}

// MN-major operand: MN columns [mn0, ...) (mn0 a multiple of 64) of a tile with
// `rows` K rows, K step s (16 rows).
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, uint32_t rows, uint32_t mn0,
                                                 uint32_t s) {
  return make_desc(base + (mn0 >> 6) * rows * 128u, rows * 128u, 1024u, kSwizzle128) +
         (uint64_t)(s * 128u);
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format,
//   13/14 negate A/B, 15/16 A/B MN-major, 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t M, uint32_t N, bool a_mn, bool b_mn,
                                                  bool negate = false) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (negate ? (1u << 13) : 0u) |
         (a_mn ? (1u << 15) : 0u) | (b_mn ? (1u << 16) : 0u) | ((N >> 3) << 17) |
         ((M >> 4) << 24);
}

// ---- mbarrier -------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
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

// Non-blocking test for the completion of phase `parity` of `bar`.
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
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

// Arrive on `bar` with `count` arrivals at once.
__device__ __forceinline__ void mbar_arrive_n(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for phase `parity` of `bar`.  Gives up after `limit_ns` of
// wall time (or at once if *abort is set), records SLIM_ERR_TIMEOUT (5) in
// *status, raises *abort for the rest of the CTA and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *status,
                                          volatile int *abort, uint64_t limit_ns = 1000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (*abort) return false;
      if (global_ns() - t0 > limit_ns) {
        atomicCAS(status, 0, 5);
        *abort = 1;
        return false;
      }
    }
  }
}

// Bounded wait that ignores the abort flag and records nothing: used only to
// let this CTA's own copies and MMAs land before it leaves.
__device__ __forceinline__ bool mbar_drain(uint64_t *bar, uint32_t parity,
                                           uint64_t limit_ns = 1000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && global_ns() - t0 > limit_ns) return false;
  }
}

// ---- TMA ------------------------------------------------------------------

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Contiguous global -> shared copy (both addresses 16-B aligned, size a
// multiple of 16), completing `bytes` of transactions on `bar`.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Contiguous shared -> global copy (16-B aligned addresses, size a multiple
// of 16) in this thread's bulk group; pair with tma_store_commit and
// tma_store_wait_read before the source may change or the CTA leaves.
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                   reinterpret_cast<uint64_t>(dst)),
               "r"(src_smem), "r"(bytes)
               : "memory");
}

// Pull a tile of a 3-D tensor map into L2 ahead of a later TMA load.
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int c0,
                                             int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_store_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Shared tile -> global tile with an add (TMA reduce-add), bulk group.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap *map, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

__device__ __forceinline__ void tma_store_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Generic-proxy smem writes -> visible to the async proxy (MMA, TMA store).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- tcgen05 --------------------------------------------------------------

// Whole warp: allocate `ncols` TMEM columns (power of two >= 32); the base
// address is written to *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A * B, issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (+)= A B with A (M = 128 rows, one per TMEM lane) in TMEM: 32-bit column
// c of a row holds the bf16 pair (k = 2c, 2c + 1), low half first, so K step
// s (16 elements) starts 8 columns on; B from shared memory.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// TMEM loads.  Each helper issues tcgen05.ld and its tcgen05.wait::ld in one
// asm statement: the loaded registers are outputs of the statement that
// waits, so no use of them can be scheduled between the load and the wait
// (with the wait in a separate statement the registers carry no dependence
// on it, and a use moved above it reads values still in flight).

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// One fp32 TMEM column of this thread's lane.
__device__ __forceinline__ float tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r)
      : "r"(taddr)
      : "memory");
  return __uint_as_float(r);
}

// Two 16-column fp32 TMEM loads of this thread's lane, one wait.
__device__ __forceinline__ void tmem_ld16x2(uint32_t a0, uint32_t a1, float *v0, float *v1) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, "
      "%27, %28, %29, %30, %31}, [%33];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(a0), "r"(a1)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v0[i] = __uint_as_float(r[i]);
    v1[i] = __uint_as_float(r[16 + i]);
  }
}

// TMEM address of (lane, column) for a base returned by tmem_alloc.
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
  return base + (lane << 16) + col;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// 8 fp32 values -> 8 bf16 -> one 16-B chunk at shared address `addr`.
__device__ __forceinline__ void st_bf16x8(uint32_t addr, const float *v) {
  st_shared_v4(addr, pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
               pack_bf16(v[6], v[7]));
}

}  // namespace tc
}  // namespace slim

namespace slim {
namespace tc {

// 16 consecutive fp32 columns into this thread's TMEM lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t &a, uint32_t &b, uint32_t &c,
                                             uint32_t &d) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
               : "r"(addr)
               : "memory");
}

// 8 bf16 at a 16-B aligned shared address -> fp32.
__device__ __forceinline__ void ld_bf16x8(uint32_t addr, float *v) {
  uint32_t w[4];
  ld_shared_v4(addr, w[0], w[1], w[2], w[3]);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

}  // namespace tc
}  // namespace slim

namespace slim {
namespace tc {

// ---- pieces shared bit-for-bit by every tensor-core kernel ------------------
// The backward recovers each tile's incoming state by removing exactly the
// values the segment pre-pass added, so the feature map and the state
// increment must round identically in both: they live here, written with
// explicit fmaf so no kernel contracts them differently.

// |x_row|^2 from a swizzled bf16 [128][D] tile.
__device__ __forceinline__ float tile_row_sqnorm(uint32_t tile_base, int row, int D) {
  // eight independent partial sums: one chain of d dependent FMAs would
  // cost d FMA latencies per row
  float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int c = 0; c < D / 8; ++c) {
    float v[8];
    ld_bf16x8(tile_base + sw128_offset(row, c * 8, 128), v);
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i] = fmaf(v[i], v[i], s[i]);
  }
  return ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
}

// Sum of squares of columns [c0, c0 + n) of a row (n a multiple of 8).
__device__ __forceinline__ float tile_row_sqnorm_part(uint32_t tile_base, int row, int c0, int n) {
  float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int c = c0; c < c0 + n; c += 8) {
    float v[8];
    ld_bf16x8(tile_base + sw128_offset(row, c, 128), v);
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i] = fmaf(v[i], v[i], s[i]);
  }
  return ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
}

// bar.sync on a named barrier (1-15) shared by `count` threads (a multiple of 32).
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

constexpr float kLog2eF = 1.4426950408889634f;

// exp2 offset of a row: phi_m = 2^(s_m log2 e + c), c = -|x|^2 log2(e)/2 - log2(sqrt(M)).
__device__ __forceinline__ float favor_row_const(float sqnorm, int M) {
  return fmaf(-0.5f * kLog2eF, sqnorm, -0.5f * log2f((float)M));
}

// 2^x on the MUFU unit (results below the fp32 normal range flush to zero;
// such features are far below bf16 resolution of any sum they enter).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float favor_feature(float s, float c) { return ex2_ftz(fmaf(s, kLog2eF, c)); }
// The same for two values: the two arguments in one packed fp32x2 FMA (each
// rounded as fmaf rounds it), then two exponentials.
__device__ __forceinline__ void favor_feature2(float &s0, float &s1, float c) {
  const float2 t = __ffma2_rn(make_float2(s0, s1), make_float2(kLog2eF, kLog2eF), make_float2(c, c));
  s0 = ex2_ftz(t.x);
  s1 = ex2_ftz(t.y);
}

__device__ __forceinline__ float elu1_feature(float x) { return x > 0.f ? x + 1.f : __expf(x); }

// no-swizzle MN-major operand of 16 columns: core matrices of 8 rows x 16 B,
// K groups of 8 rows 256 B apart, the two 8-column groups 128 B apart.
__host__ __device__ __forceinline__ uint32_t n16_offset(uint32_t k, uint32_t n) {
  return (n >> 3) * 128u + (k >> 3) * 256u + (k & 7u) * 16u + (n & 7u) * 2u;
}

__device__ __forceinline__ uint64_t desc_n16(uint32_t base, uint32_t s) {
  return make_desc(base, 256u, 128u, 0u) + (uint64_t)(s * 32u);
}

// Increment of one 128-feature block of R'^T over one tile:
//   delta[f][e] = sum_j phi_k[j][f] V'[j][e],  V' = [V, 1]   (columns 0..D)
// issued by one thread; `phk` is the [128][128] swizzled phi_k tile (block
// features in columns 0..127), `v` the [128][D] V tile, `ones` the 16-column
// ones operand.  Accumulation restarts at zero, so the result depends only
// on the operands.
__device__ __forceinline__ void issue_state_delta(uint32_t t_delta, uint32_t phk, uint32_t v,
                                                  uint32_t ones, int D) {
  const uint32_t id = make_idesc(128, D, true, true);
  const uint32_t id1 = make_idesc(128, 16, true, true);
  for (int s = 0; s < 8; ++s) {
    mma_bf16(t_delta, desc_mnmajor(phk, 128, 0, s), desc_mnmajor(v, 128, 0, s), id, s > 0);
    mma_bf16(t_delta + D, desc_mnmajor(phk, 128, 0, s), desc_n16(ones, s), id1, s > 0);
  }
}

// (hi, lo) += sign * x as a double-float (two-sum, then renormalise).
__device__ __forceinline__ void df_add(float &hi, float &lo, float x) {
  const float s = hi + x;
  const float bp = s - hi;
  const float e = (hi - (s - bp)) + (x - bp);
  const float t = lo + e;
  hi = s + t;
  lo = t - (hi - s);
}

// df_add(hi, lo, -x) for two values at once in packed fp32x2 arithmetic,
// bit for bit: a - b is formed as fma(b, -1, a), which rounds the exact
// difference once, as the subtraction does.
__device__ __forceinline__ void df_sub2(float2 &hi, float2 &lo, float2 x) {
  const float2 m1 = make_float2(-1.f, -1.f);
  const float2 s = __ffma2_rn(x, m1, hi);                          // hi - x
  const float2 bp = __ffma2_rn(hi, m1, s);                         // s - hi
  const float2 e1 = __ffma2_rn(__ffma2_rn(bp, m1, s), m1, hi);     // hi - (s - bp)
  const float2 e = __ffma2_rn(__fadd2_rn(x, bp), m1, e1);          // e1 + (-x - bp)
  const float2 t = __fadd2_rn(lo, e);
  hi = __fadd2_rn(s, t);
  lo = __ffma2_rn(__ffma2_rn(s, m1, hi), m1, t);                   // t - (hi - s)
}

// Columns [c_lo, c_hi) (multiples of 16) of this warp's 32 lanes:
// (hi, lo) += sign * delta, all three in TMEM.
__device__ __forceinline__ void df_update_tmem(uint32_t tbase, int lane_base, uint32_t t_delta,
                                               uint32_t t_hi, uint32_t t_lo, int c_lo, int c_hi,
                                               float sign) {
  for (int c = c_lo; c < c_hi; c += 16) {
    float x[16], h[16], l[16];
    tmem_ld16(tmem_addr(tbase, lane_base, t_delta + c), x);
    tmem_ld16(tmem_addr(tbase, lane_base, t_hi + c), h);
    tmem_ld16(tmem_addr(tbase, lane_base, t_lo + c), l);
#pragma unroll
    for (int i = 0; i < 16; ++i) df_add(h[i], l[i], sign * x[i]);
    tmem_st16(tmem_addr(tbase, lane_base, t_hi + c), h);
    tmem_st16(tmem_addr(tbase, lane_base, t_lo + c), l);
  }
  tmem_st_wait();
}

}  // namespace tc
}  // namespace slim

namespace slim {
namespace tc {

// ---- thread-block clusters (distributed shared memory) ----------------------

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared address of the same offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_peer(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_peer_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

__device__ __forceinline__ void st_peer_v4u(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                            uint32_t d) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b),
               "r"(c), "r"(d)
               : "memory");
}

// Fire-and-forget add of four consecutive floats into global memory.
__device__ __forceinline__ void red_add_v4(float *addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

__device__ __forceinline__ void st_peer_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void st_peer_b16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared::cluster.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// Store to a peer CTA's shared memory (cluster address) that completes
// its bytes as transactions on the peer's mbarrier `rbar` (cluster address).
__device__ __forceinline__ void st_async_v4(uint32_t addr, float a, float b, float c, float d,
                                            uint32_t rbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
      "f"(a), "f"(b), "f"(c), "f"(d), "r"(rbar)
      : "memory");
}

__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(addr), "f"(v),
               "r"(rbar)
               : "memory");
}

// Arrive (release, cluster scope) on an mbarrier of a peer CTA.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t rbar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(rbar) : "memory");
}

// All threads of every CTA in the cluster; orders shared (incl. remote) and
// global memory like __syncthreads does within a CTA.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void ld_shared_v4f(uint32_t addr, float *v) {
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
               : "r"(addr)
               : "memory");
}

}  // namespace tc
}  // namespace slim

namespace slim {
namespace tc {

// Two 32-column TMEM loads (any two addresses of this warp's lanes) with a
// single wait, so their latencies overlap.
__device__ __forceinline__ void tmem_ld32x2(uint32_t a0, uint32_t a1, float *v0, float *v1) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, "
      "%42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, "
      "%60, %61, %62, %63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]),
        "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]),
        "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]),
        "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]),
        "=r"(r[62]), "=r"(r[63])
      : "r"(a0), "r"(a1)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v0[i] = __uint_as_float(r[i]);
    v1[i] = __uint_as_float(r[32 + i]);
  }
}

// Three 16-column TMEM loads with a single wait.
__device__ __forceinline__ void tmem_ld16x3(uint32_t a0, uint32_t a1, uint32_t a2, float *v0, float *v1,
                                            float *v2) {
  uint32_t r[48];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%48];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, "
      "%26, %27, %28, %29, %30, %31}, [%49];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, "
      "%42, %43, %44, %45, %46, %47}, [%50];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47])
      : "r"(a0), "r"(a1), "r"(a2)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v0[i] = __uint_as_float(r[i]);
    v1[i] = __uint_as_float(r[16 + i]);
    v2[i] = __uint_as_float(r[32 + i]);
  }
}

// Three single-column TMEM loads with a single wait.
__device__ __forceinline__ void tmem_ld1x3(uint32_t a0, uint32_t a1, uint32_t a2, float &v0, float &v1,
                                           float &v2) {
  uint32_t r0, r1, r2;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%3];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%1}, [%4];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%2}, [%5];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r0), "=r"(r1), "=r"(r2)
      : "r"(a0), "r"(a1), "r"(a2)
      : "memory");
  v0 = __uint_as_float(r0);
  v1 = __uint_as_float(r1);
  v2 = __uint_as_float(r2);
}

// One fp32 column into this thread's TMEM lane.
__device__ __forceinline__ void tmem_st1(uint32_t taddr, float v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(__float_as_uint(v)) : "memory");
}

// A 32-column and a 16-column TMEM load with a single wait.
__device__ __forceinline__ void tmem_ld32p16(uint32_t a0, uint32_t a1, float *v0, float *v1) {
  uint32_t r[48];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%48];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, "
      "%42, %43, %44, %45, %46, %47}, [%49];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47])
      : "r"(a0), "r"(a1)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v0[i] = __uint_as_float(r[i]);
#pragma unroll
  for (int i = 0; i < 16; ++i) v1[i] = __uint_as_float(r[32 + i]);
}

// 8 consecutive fp32 columns into this thread's TMEM lane.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float *v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
               "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
               : "memory");
}

}  // namespace tc
}  // namespace slim
