// Blackwell (sm_100-family) tensor-core helpers written against the public
// PTX ISA: tcgen05 MMA with operands in shared memory, accumulators in tensor
// memory (TMEM), completion through an mbarrier.
//
// Operand layout used everywhere in this library: "K-major, 128-byte swizzle".
// A tile of R rows (R a multiple of 8) and K bf16 columns is stored as K/64
// blocks of R x 128 bytes; inside a block, row r occupies 128 bytes at
// (r / 8) * 1024 + (r % 8) * 128 and its 16-byte chunk c sits at chunk
// position c ^ (r % 8).  Tiles must start on a 1024-byte boundary.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace kda {
namespace umma {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The first 1024-byte aligned byte of a dynamic shared-memory array, reached
// by an offset from the array itself rather than through an integer, so the
// compiler still knows that pointers derived from it address shared memory.
__device__ __forceinline__ unsigned char *align1024(void *smem) {
  unsigned char *b = static_cast<unsigned char *>(smem);
  return b + ((1024u - (smem_u32(b) & 1023u)) & 1023u);
}

// Shared-memory matrix descriptor: start address, leading byte offset (unused
// for swizzled K-major tiles), stride byte offset between 8-row groups
// (1024), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFF) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Descriptor of an MN-major operand with the 128-byte swizzle: K-rows of
// 128 bytes (64 MN elements, one atom), 8-row groups 1024 bytes apart, and
// atoms along MN `atom_stride` bytes apart (the leading byte offset; unused
// when the operand's MN extent is a single atom).
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t addr, uint32_t atom_stride = 1024) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFF) >> 4);
  d |= (uint64_t)((atom_stride >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Byte offset of element (k, n) of such an MN-major tile (n < 64): K-row k
// holds n = 0..63 contiguous, 16-byte chunks swizzled by k % 8.
__host__ __device__ __forceinline__ uint32_t sw128_mn_off16(int k, int n) {
  return (uint32_t)((k >> 3) * 1024 + (k & 7) * 128 + ((((n >> 3) ^ (k & 7))) << 4) +
                    (n & 7) * 2);
}

// Byte offset of element (row, k) of a K-major SW128 tile of 16-bit elements
// with `rows` rows: K/64 blocks of rows x 128 bytes, 8 elements per 16-byte
// chunk, swizzled as above.
__host__ __device__ __forceinline__ uint32_t sw128_off16(int row, int k, int rows) {
  const int kb = k >> 6, kin = k & 63;
  const int chunk = kin >> 3, within = kin & 7;
  const int r8 = row & 7;
  return (uint32_t)(kb * rows * 128 + (row >> 3) * 1024 + r8 * 128 +
                    ((chunk ^ r8) << 4) + within * 2);
}

// Instruction descriptor: kind::f16 with bf16 A and B, fp32 accumulator,
// A and B K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
// The same with B MN-major (bit 16: B transposed), and with A and B MN-major
// (bit 15: A transposed).
__host__ __device__ constexpr uint32_t idesc_bf16_bmn(int M, int N) {
  return idesc_bf16(M, N) | (1u << 16);
}
__host__ __device__ constexpr uint32_t idesc_bf16_abmn(int M, int N) {
  return idesc_bf16(M, N) | (1u << 15) | (1u << 16);
}

// D (TMEM) (+)= A * B^T for one K = 16 step; A is M x 16, B is N x 16 (bf16).
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t da,
                                         uint64_t db, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(da), "l"(db), "r"(idesc), "r"(accumulate));
}

// Two fp32 values as bf16 pairs hi + lo with hi = rn(x), lo = rn(x - hi):
// hi + lo carries 16 significant bits, and the three products hi*hi,
// hi*lo, lo*hi of two such splits reproduce an fp32 product to ~2^-16.
// The first value goes to the low half of each word (lower address).
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t &hi,
                                             uint32_t &lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  lo = *reinterpret_cast<const uint32_t *>(&l);
}
__device__ __forceinline__ void split_bf16(float x, uint16_t &hi, uint16_t &lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
  hi = __bfloat16_as_ushort(h);
  lo = __bfloat16_as_ushort(l);
}

// Arrive on `mbar` once every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void commit(uint64_t *mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
      :: "r"(smem_u32(mbar)) : "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t *mbar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;"
               :: "r"(smem_u32(mbar)), "r"(count));
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from global into shared memory, completing on `mbar`'s transaction count.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1], %2, [%3];"
      :: "r"(dst), "l"(src), "r"(bytes), "r"(mbar) : "memory");
}
// Bulk copy from shared into global memory (same rules), in the issuing
// thread's current bulk group.
__device__ __forceinline__ void bulk_s2g(void *dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               :: "l"(dst), "r"(src), "r"(bytes) : "memory");
}
// Close the issuing thread's bulk group, and wait until every group it
// closed has finished reading shared memory.
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Hint: bring `bytes` (a multiple of 16) at `src` into L2.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(src), "r"(bytes)
               : "memory");
}

// Wait for phase `parity` of `mbar` to complete; gives up after `limit`
// polls and returns false (the caller reports a device error).
__device__ __forceinline__ bool mbar_wait(uint64_t *mbar, uint32_t parity,
                                          int limit) {
  uint32_t done = 0;
  for (int it = 0; it < limit; ++it) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(smem_u32(mbar)), "r"(parity) : "memory");
    if (done) return true;
  }
  return false;
}

// Warp-collective TMEM allocation of `ncols` columns (power of two >= 32);
// the TMEM address is written to *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(smem_u32(slot)), "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
               :: "r"(taddr), "r"(ncols));
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to the
// tensor core (async proxy).
__device__ __forceinline__ void fence_smem_to_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16 consecutive TMEM columns of this thread's lane -> registers.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive TMEM columns of this thread's lane -> registers (one load,
// one wait).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
        "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]),
                 "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]),
                 "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive TMEM columns -> registers without waiting (see tmem_wait16).
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// Waits for this thread's TMEM loads.  The destination registers of the
// loads pass through the wait, so no use of them is placed before it.
__device__ __forceinline__ void tmem_wait16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :: "memory");
}
// Ties further loads' registers to a wait already done (an empty statement
// with the same effect on ordering: nothing reads them before this point,
// which follows the wait).
__device__ __forceinline__ void tmem_tie16(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :: "memory");
}
// Sums of pairs of 16-column TMEM loads issued together and waited for once:
// x[i] = a[i] + b[i] (the hi and lo halves of one accumulator).
__device__ __forceinline__ void tmem_ld16_pair_sum(uint32_t ta, uint32_t tb, float (&x)[16]) {
  uint32_t a[16], b[16];
  tmem_ld16_nowait(ta, a);
  tmem_ld16_nowait(tb, b);
  tmem_wait16(a);
  tmem_tie16(b);
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = __uint_as_float(a[i]) + __uint_as_float(b[i]);
}
// Two such pair sums with one wait.
__device__ __forceinline__ void tmem_ld16_pair_sum2(uint32_t ta, uint32_t tb, uint32_t tc,
                                                    uint32_t td, float (&x)[16],
                                                    float (&y)[16]) {
  uint32_t a[16], b[16], c[16], d[16];
  tmem_ld16_nowait(ta, a);
  tmem_ld16_nowait(tb, b);
  tmem_ld16_nowait(tc, c);
  tmem_ld16_nowait(td, d);
  tmem_wait16(a);
  tmem_tie16(b);
  tmem_tie16(c);
  tmem_tie16(d);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    x[i] = __uint_as_float(a[i]) + __uint_as_float(b[i]);
    y[i] = __uint_as_float(c[i]) + __uint_as_float(d[i]);
  }
}

// 8 consecutive TMEM columns -> registers without waiting; the values are
// valid only after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld8_async(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

}  // namespace umma
}  // namespace kda
