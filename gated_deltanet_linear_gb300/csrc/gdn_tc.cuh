// Blackwell (sm_100-family) tensor-core primitives used by the chunked
// prefill: tcgen05 MMA with operands in shared memory and the accumulator in
// tensor memory (TMEM), completion tracked by mbarriers, TMEM <-> register
// moves.  Inline PTX only.
//
// Operand tiles are K-major with the 128-byte swizzle: a tile of R rows and
// K elements is stored as K / (128 / elem_bytes) column blocks, each block
// R rows x 128 bytes, rows consecutive; inside a block, 16-byte chunk c of
// row r is stored at chunk position c ^ (r & 7).  Blocks start on 1024-byte
// boundaries.  One MMA consumes 32 bytes of K per row (16 bf16 elements),
// so the descriptor start steps by 32 bytes within a block.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {
namespace tc {

// ----------------------------------------------------------- descriptors

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);  // start address >> 4
  d |= (uint64_t)1 << 16;                         // leading byte offset (unused)
  d |= (uint64_t)(1024 >> 4) << 32;               // stride byte offset >> 4
  d |= (uint64_t)1 << 46;                         // version
  d |= (uint64_t)2 << 61;                         // layout: 128-byte swizzle
  return d;
}

enum : uint32_t { kFmtBF16 = 1 };

// Instruction descriptor: fp32 accumulator, A and B of format `fmt`, both
// K-major, M x N tile.
__host__ __device__ constexpr uint32_t idesc(uint32_t fmt, int M, int N) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------------------ MMA

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a,
                                         uint64_t b, uint32_t id,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(accumulate));
}

// The same product with A in tensor memory: A's row m is TMEM lane m, and
// its K elements are packed two bf16 per 32-bit column (the lower index in
// the low half), so one K step of 16 elements is 8 columns.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem,
                                            uint64_t b, uint32_t id,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate));
}

// Arrive on the mbarrier once every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void commit(uint32_t mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];" ::"r"(mbar)
      : "memory");
}

// ----------------------------------------------------------------- TMEM

// Allocate ncols (power of two, 32..512) columns; the TMEM address is written
// to shared memory at `dst`.  Whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile(
      "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
          dst),
      "r"(ncols)
      : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(
                   taddr),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (the tensor cores).
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32 lanes x 16 columns of 32-bit values: thread t of the warp receives lane
// (base lane + t), columns col .. col+15.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&r)[16]) {
  uint32_t u[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]),
        "=r"(u[5]), "=r"(u[6]), "=r"(u[7]), "=r"(u[8]), "=r"(u[9]),
        "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]),
        "=r"(u[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) r[i] = __uint_as_float(u[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16};" ::"r"(taddr),
      "r"(__float_as_uint(r[0])), "r"(__float_as_uint(r[1])),
      "r"(__float_as_uint(r[2])), "r"(__float_as_uint(r[3])),
      "r"(__float_as_uint(r[4])), "r"(__float_as_uint(r[5])),
      "r"(__float_as_uint(r[6])), "r"(__float_as_uint(r[7])),
      "r"(__float_as_uint(r[8])), "r"(__float_as_uint(r[9])),
      "r"(__float_as_uint(r[10])), "r"(__float_as_uint(r[11])),
      "r"(__float_as_uint(r[12])), "r"(__float_as_uint(r[13])),
      "r"(__float_as_uint(r[14])), "r"(__float_as_uint(r[15]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 8 columns of 32-bit values from registers, without waiting for
// completion (tmem_wait_st does, before the values are used elsewhere).
__device__ __forceinline__ void tmem_st8_async(uint32_t taddr, const uint32_t (&u)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, "
      "%8};" ::"r"(taddr),
      "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]),
      "r"(u[6]), "r"(u[7])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mbar),
               "r"(count)
               : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Wait for the phase with the given parity to complete; gives up after
// `limit` polls and returns false (the caller records the failure).
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity,
                                          uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(mbar), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}

// ------------------------------------------------- operand tile layout

// Byte offset of element (r, k) in a K-major 128-byte-swizzled tile of R
// rows whose elements are `eb` bytes.
__device__ __forceinline__ uint32_t sw128_off(int R, int r, int k, int eb) {
  const int per_block = 128 / eb;
  const int kb = k / per_block;
  const int kin = k % per_block;
  const int chunk = (kin * eb) >> 4;
  const int within = (kin * eb) & 15;
  return (uint32_t)(kb * R * 128 + r * 128 + ((chunk ^ (r & 7)) << 4) + within);
}

// Descriptor of K step `ks` (32 bytes of K) of a tile of R rows at `base`.
__device__ __forceinline__ uint64_t desc_kstep(uint32_t base, int R, int ks) {
  return desc_sw128(base + (uint32_t)((ks >> 2) * R * 128 + (ks & 3) * 32));
}

}  // namespace tc
}  // namespace gdn
