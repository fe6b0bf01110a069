// Thin inline-PTX wrappers for the sm_100-family tensor-core path used by the
// chunked scan: TMEM allocation, tcgen05.mma (kind::tf32) with shared-memory
// and tensor-memory operands, tcgen05.commit to an mbarrier, TMEM loads and
// stores, and bounded mbarrier waits.
//
// Operand tiles in shared memory use the canonical K-major layout without
// swizzling: a tile of `rows` x `kext` 32-bit elements is made of 8-row x
// 16-byte core matrices (128 contiguous bytes); core matrices adjacent along K
// are 128 B apart (descriptor leading-byte offset) and 8-row groups are
// kext * 32 B apart (descriptor stride-byte offset).
#pragma once

#include <stdint.h>

namespace m3 {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Float offset of element (row, k) in a K-major tile whose K extent is kext.
__device__ __forceinline__ int kmaj(int row, int k, int kext) {
  return (((row >> 3) * (kext >> 2) + (k >> 2)) << 5) + ((row & 7) << 2) + (k & 3);
}

// Float offset of element (row, k) in a K-major tile with the 128-byte swizzle
// (the layout a TMA tile copy with CU_TENSOR_MAP_SWIZZLE_128B writes): K is
// cut into column blocks of 32 elements; a block holds `rows` rows of 128 B,
// and the 16-byte chunk c of row r sits at chunk position c ^ (r % 8). The
// tile must start on a 1024-byte boundary.
__device__ __forceinline__ int sw128(int row, int k, int rows) {
  return (((k >> 5) * rows + row) << 5) + ((((k & 31) >> 2) ^ (row & 7)) << 2) + (k & 3);
}

// Shared-memory matrix descriptor (no swizzle, sm_100 descriptor version 1).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// Descriptor of a K-major tile with K extent kext, advanced by kstep groups of
// 8 elements (one MMA K step = two core matrices = 256 B).
__device__ __forceinline__ uint64_t kdesc(const float* tile, int kext, int kstep) {
  return sdesc(smem_u32(tile) + (uint32_t)kstep * 256u, 128u, (uint32_t)kext * 32u);
}
// Descriptor of a K-major 128-byte-swizzled tile (layout of sw128): 8-row
// atoms of 1024 B along M / N (stride-byte offset 1024), swizzle mode 2 in
// bits 61..63. One MMA K step (8 elements = 32 B) advances the start address
// by 32 B inside a 128-byte row; the next column block starts rows * 128 B on.
__device__ __forceinline__ uint64_t swdesc(const float* tile) {
  return sdesc(smem_u32(tile), 16u, 1024u) | (2ull << 61);
}
__host__ __device__ constexpr uint32_t swdesc_kstep(int ks, int rows) {
  return (uint32_t)(((ks >> 2) * rows * 128 + (ks & 3) * 32) >> 4);  // in descriptor units
}

// Instruction descriptor: kind::tf32, dense, D = F32, A = B = TF32, A
// K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1, bit 16), N >> 3 at
// bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N, int b_mn = 0) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// L2 prefetch of a byte range (start and size multiples of 16 bytes).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar)));
}

__device__ __forceinline__ void bar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
// One wait attempt; the thread may stay suspended for up to about 0.1 ms
// (suspend-time hint, in ns) unless the phase completes first, so that waiting
// threads do not spin through issue slots.
__device__ __forceinline__ bool bar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(100000u));
  return ok != 0;
}
// Bounded wait: false once about `budget` clock cycles have passed.
__device__ __forceinline__ bool bar_wait(uint64_t* bar, uint32_t parity, long long budget) {
  const long long t0 = clock64();
  while (!bar_try(bar, parity)) {
    if (clock64() - t0 > budget) return false;
  }
  return true;
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;"); }
// Makes generic-proxy shared-memory writes visible to the tensor core.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;"); }

// Warp-collective TMEM allocation (result written to *slot) and release.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_free(uint32_t base, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols));
}

// 32 lanes x 16 consecutive 32-bit columns: thread i of the warp gets lane
// (warp quadrant base + i). Includes the wait.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])));
}

// TMA: 4-D tiled copy of one box of the tensor map into shared memory,
// completing `bytes` of transaction count on the mbarrier (coordinates are
// element indices, innermost first).
__device__ __forceinline__ void tma_load_4d(void* dst, const void* tmap, int c0, int c1, int c2,
                                           int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}
// Arrives on the mbarrier and raises its expected transaction count.
__device__ __forceinline__ void bar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Two 32-lane x 16-column loads with a single wait (fewer serialised waits).
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, float* va, float* vb) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(ta), "r"(tb));
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    va[i] = __uint_as_float(r[i]);
    vb[i] = __uint_as_float(r[16 + i]);
  }
}
// M = 64 accumulator tiles (cta_group::1) keep their 64 rows in lanes 0..15
// of each 32-lane quadrant. The .16x32bx2 shape reads those 16 lanes twice:
// threads 0..15 get columns [c, c + n) of lanes 0..15, threads 16..31 the
// columns [c + off, c + off + n) of the same lanes, so every thread holds
// useful data.
// Two 8-column half-split loads (off = 8), one wait: va = columns [ca + 8h,
// ca + 8h + 8) and vb likewise at cb, where h = thread / 16.
__device__ __forceinline__ void tmem_ld_m64_8x2(uint32_t ta, uint32_t tb, float* va, float* vb) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%16], 8;\n\t"
      "tcgen05.ld.sync.aligned.16x32bx2.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%17], 8;\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(ta), "r"(tb));
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    va[i] = __uint_as_float(r[i]);
    vb[i] = __uint_as_float(r[8 + i]);
  }
}
// One 16-column half-split load (off = 16): v = columns [c + 16h, c + 16h + 16),
// h = thread / 16, so a warp covers 32 columns of its 16 rows. No wait.
__device__ __forceinline__ void tmem_ld_m64_16(uint32_t ta, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16], 16;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(ta));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// The matching store (no wait).
__device__ __forceinline__ void tmem_st_m64_16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x16.b32 [%0], 16, {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}

// Store without waiting; tmem_wait_st() before the data is handed to an MMA.
__device__ __forceinline__ void tmem_st16_async(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// TF32 operand rounding. A kind::tf32 MMA reads the sign, the exponent and the
// top 10 mantissa bits of each 32-bit element and ignores the low 13 bits, so
// adding half a TF32 unit in the last place (0x1000) to the bit pattern makes
// the MMA see the value rounded to nearest (ties away from zero) at the cost of
// one integer add. tf32_feed is for values that only the tensor core reads;
// tf32_clean also clears the ignored bits, for values that are read back as
// FP32 as well. Both turn an infinity into a NaN.
__device__ __forceinline__ float tf32_feed(float v) {
  return __uint_as_float(__float_as_uint(v) + 0x1000u);
}
__device__ __forceinline__ float4 tf32_feed(float4 v) {
  return make_float4(tf32_feed(v.x), tf32_feed(v.y), tf32_feed(v.z), tf32_feed(v.w));
}
__device__ __forceinline__ float tf32_clean(float v) {
  return __uint_as_float((__float_as_uint(v) + 0x1000u) & 0xFFFFE000u);
}
// The value as a kind::tf32 MMA reads an unrounded operand (low 13 bits dropped).
__device__ __forceinline__ float tf32_trunc(float v) {
  return __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
}

}  // namespace tc
}  // namespace m3
