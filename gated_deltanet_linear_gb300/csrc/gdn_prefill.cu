// Chunk-parallel prefill of the gated delta rule on tcgen05 tensor cores.
//
// The token-serial definition ("Kestrel_VLLM - 24 · GDN linear attention to
// GPU", section 4) is regrouped into chunks of C = 64 tokens.  The articles
// process tokens strictly one after another ("34 · batched M rows",
// section 3.6, no chunked scan); the chunked form below follows from that
// recurrence.  Within a chunk starting from state S0 (kd x vd), with
// Gamma_t = sum_{s<=t} g_s, gamma_t = exp(Gamma_t), w_t = exp(Gamma_63 -
// Gamma_t):
//   A[t,s] = beta_t exp(Gamma_t - Gamma_s) k_t.k_s   (s < t),  T = (I + A)^-1
//   W = T diag(beta gamma) K,   U = T diag(beta) V
//   Delta = U - W S0                      (the per-token corrections)
//   O = diag(gamma) Q S0 + P Delta,  P[t,s] = exp(Gamma_t - Gamma_s) q_t.k_s (s <= t)
//   S_C = gamma_63 S0 + (diag(w) K)^T Delta
//
// One CTA per (sequence, value head) walks the chunks in order; the fp32
// state is kept transposed (S^T: one TMEM lane per value column dv, one
// column per key row dk) in tensor memory for the whole sequence.  Since
// (W S)^T = S^T W^T = (S^T K^T) (T diag(beta gamma))^T, the two products
// with the chunk-start state, Y = S^T K^T and (Q S)^T = S^T Q^T, need only
// that state and the chunk's inputs: they are issued early and run under
// the SIMT work on A and its inverse.  Per chunk (D = M x N accumulator in
// TMEM, lanes = M):
//   MMA-a  G,H  [t'][s]  = [K; Q] K^T                       (A, B K-major)
//   SIMT   S^T operand, then S^T *= gamma_63, both in TMEM (under MMA-a)
//   MMA-s  [Y | (Q S)^T] [dv][t'] = S^T [K; Q]^T      (one N = 128 product)
//   SIMT   o of the previous chunk;  A and P from G, H;
//          T = (I + A)^-1, blocked 16 x 16, fp32 (under MMA-s)
//   SIMT   V^T - Y diag(gamma) operand in TMEM; T diag(beta) operand
//   MMA-ud Delta^T [dv][t] = (V^T - Y diag(gamma)) (T diag(beta))^T
//          (= U^T - (W S)^T in one product)
//   SIMT   Delta^T and Delta^T diag(w) operands in TMEM
//   MMA-3  (P Delta)^T = Delta^T P^T
//   MMA-4  S^T += (Delta^T diag(w)) K                        (B = K, MN-major)
//   SIMT   O^T = diag(gamma) (Q S)^T + (P Delta)^T  -> o, emitted in the
//          next chunk while its first products run
// Every operand a thread writes is a row it owns: a row of an input, stored
// in shared memory 8 elements at a time, or a TMEM lane of an earlier
// result, which stays in its lane as an A operand in TMEM (S^T,
// V^T - Y diag(gamma), Delta^T); transposes happen in the MMA descriptors
// (MN-major operands), never in memory.  Every input tile arrives by tensor
// copy a chunk ahead: K and Q into a region of their own per chunk parity,
// where the next chunk's [K; Q] operand is made in place while the current
// chunk's last products run; V into its region once the previous chunk's
// rows are read.  The gates come through registers.
//
// Precision.  Operands are bf16 in shared memory:
//   split-bf16 ("BF16X3"): x = hi + lo with hi = bf16(x), lo = bf16(x - hi);
//     a product is hi*hi + hi*lo + lo*hi, three MMAs with fp32 accumulation
//     (about 16 significant bits per operand; ~1e-5 relative error);
//   plain bf16: hi only, one MMA per product (~1e-2 relative error).
// The triangular solve, the gating exponentials and every accumulation are
// fp32.

#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gdn_internal.cuh"
#include "gdn_tc.cuh"

namespace gdn {

__device__ unsigned int g_prefill_timeouts = 0;

namespace {

using namespace tc;

constexpr int kC = 64;       // chunk length
constexpr int kD = kDim;     // 128
constexpr int kSimt = 256;              // 8 SIMT warps
constexpr int kIssuer = kSimt / 32;     // warp that issues the products
constexpr int kLoader = kIssuer + 1;    // warp that copies the next K, Q
constexpr int kThreads = kSimt + 64;

// Operand tiles: R rows x C bf16 columns, 128-byte-swizzled blocks of 64
// columns (see gdn_tc.cuh), hi tile followed by lo tile (R * C * 2 bytes
// each).  Regions (byte offsets from a 1024-aligned base) are reused by
// phase:
//   Ra 64 KB: even chunks' K, Q rows: fp32 staging, converted in place
//             (read, barrier, write) to the [K; Q] operand (128 x 128)
//   Rb 32 KB: fp32 V rows of the chunk
//   Rc 32 KB: o of the previous chunk (fp32 [t][dv], 64 x 128, read by a
//             tensor store before the A build)
//                                     -> A, T scratch (fp32)
//                                     -> T diag(beta) (64 x 64) over the
//                                        A half, while T is still read
//   Rd 64 KB: the same for odd chunks, so a chunk's K, Q arrive and are
//             converted while the previous chunk still reads its own
//   Rp 16 KB: P (64 x 64)
// The operands made from TMEM results (S^T, Y, Delta^T) stay in TMEM.
constexpr uint32_t RA = 0, RB = 65536, RC = 98304, RD = 131072, RP = 196608;
// [K; Q] region of chunk c: fp32 staging, then the 128 x 128 operand
__host__ __device__ constexpr uint32_t kq_region(int c) { return (c & 1) ? RD : RA; }
constexpr uint32_t OFF_V = RB;              // fp32 V rows [64][128]
constexpr uint32_t OFF_OT = RC;             // fp32 o tile [64][128]
constexpr uint32_t OFF_SCR = RC;            // fp32 A [64][64] + T [64][64]
constexpr uint32_t OFF_TB2 = RC;            // 64 x 64: T diag(beta), over A
constexpr uint32_t OFF_P = RP;              // 64 x 64
// Gate vectors of chunk c in buffer c & 1, 512 floats: Gamma +0, gamma +64,
// w +128, beta +192, ea +384, eb +448.
constexpr uint32_t OFF_VEC = RP + 16384;      // buffer 0
constexpr uint32_t OFF_BAR = OFF_VEC + 2048;  // 14 mbarriers
constexpr uint32_t OFF_SLOT = OFF_BAR + 112;  // TMEM address; +120: int flags
constexpr uint32_t OFF_VEC1 = OFF_BAR + 128;  // buffer 1
constexpr uint32_t kSmemUsed = OFF_VEC1 + 2048;
constexpr uint32_t kSmemAlloc = kSmemUsed + 1024;  // room to align the base

// TMEM columns (512 allocated).
constexpr uint32_t T_SACC = 0;    // S^T: lanes dv, 128 columns dk
constexpr uint32_t T_GH = 128;    // G (lanes 0-63), H (lanes 64-127): 64 columns
constexpr uint32_t T_U = 192;     // second half-K of G, H; then
                                  // Delta^T = U^T - (W S)^T: lanes dv
// 128 columns, lanes dv, columns t: MMA-s writes [Y | (Q S)^T] in one
// product (B = [K; Q]); once Y has been read out, MMA-3 writes
// (P Delta)^T over it, and the next chunk reads [(P Delta)^T | (Q S)^T]
// for the output before its own MMA-s is issued.
constexpr uint32_t T_BUF = 256;
// 128 columns of bf16 A operands (lanes dv, two elements per column), hi
// then lo: S^T (64 + 64 columns, K = dk) for MMA-s; then V^T - Y diag(gamma)
// (32 + 32, K = t) for MMA-ud; then Delta^T (32 + 32) and Delta^T diag(w)
// (the next 64) for MMA-3 and MMA-4.
constexpr uint32_t T_AOP = 384;

constexpr uint32_t kWaitLimit = 1u << 24;

// ----------------------------------------------------------- operands

__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 v) {
  return *reinterpret_cast<uint32_t *>(&v);
}

// Store columns c0..c0+7 (c0 % 8 == 0) of row r of an R x C tile.
template <bool kLo>
__device__ __forceinline__ void put8(unsigned char *gb, uint32_t off, int R,
                                     int C, int r, int c0, const float *x) {
  uint32_t hi[4], lo[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
    hi[i] = bf2_bits(h);
    if (kLo) {
      const float2 f = __bfloat1622float2(h);
      lo[i] = bf2_bits(__floats2bfloat162_rn(x[2 * i] - f.x, x[2 * i + 1] - f.y));
    }
  }
  const uint32_t o = off + sw128_off(R, r, c0, 2);
  *reinterpret_cast<uint4 *>(gb + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  if (kLo)
    *reinterpret_cast<uint4 *>(gb + o + (uint32_t)(R * C * 2)) =
        make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

// Columns c0 .. c0+15 (c0 % 16 == 0) of this thread's lane of a bf16 A
// operand in tensor memory whose hi part starts at TMEM address `hi` and lo
// part at `lo` (both including the lane): two elements per 32-bit column.
// The stores are asynchronous; tmem_wait_st completes them.
template <bool kLo>
__device__ __forceinline__ void put16_tmem(uint32_t hi, uint32_t lo, int c0,
                                           const float *x) {
  uint32_t h[8], l[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
    h[i] = bf2_bits(v);
    if (kLo) {
      const float2 f = __bfloat1622float2(v);
      l[i] = bf2_bits(__floats2bfloat162_rn(x[2 * i] - f.x, x[2 * i + 1] - f.y));
    }
  }
  tmem_st8_async(hi + (uint32_t)(c0 >> 1), h);
  if (kLo) tmem_st8_async(lo + (uint32_t)(c0 >> 1), l);
}

// Shared-memory descriptor of K step ks (16 bf16 of K) of a tile:
//   K-major: rows are the M (or N) index, columns the K index.
//   MN-major: rows are the K index, columns the M (or N) index; 64-column
//   blocks are R * 128 bytes apart (leading byte offset), 8-row groups
//   1024 bytes apart (stride byte offset), one K step = 16 rows.
__device__ __forceinline__ uint64_t kmajor(uint32_t base, int R, int ks) {
  return desc_kstep(base, R, ks);
}

__device__ __forceinline__ uint64_t mnmajor(uint32_t base, int R, int ks) {
  uint64_t d = desc_sw128(base + (uint32_t)ks * 2048u);
  d &= ~((uint64_t)0x3FFF << 16);
  d |= (uint64_t)(((uint32_t)R * 128u) >> 4) << 16;
  return d;
}

__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn,
                                                  int b_mn) {
  return idesc(kFmtBF16, M, N) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16);
}

struct Operand {
  uint32_t base;  // hi tile (shared address)
  int R, C;       // tile shape
  bool mn;        // MN-major use
};

// Descriptor of K step 0 of the hi (lo = false) or lo tile of an operand.
__device__ __forceinline__ uint64_t opdesc(const Operand &o, bool lo) {
  const uint32_t base = o.base + (lo ? (uint32_t)(o.R * o.C * 2) : 0u);
  return o.mn ? mnmajor(base, o.R, 0) : kmajor(base, o.R, 0);
}

// Start-address step of K step ks, in the descriptor's 16-byte units.  The
// start address is the descriptor's low field (shared address >> 4, 14
// bits; every tile lies below 256 KB), so the descriptor of K step ks is
// the K-step-0 descriptor plus this constant.
__device__ __forceinline__ uint32_t kstep16(const Operand &o, int ks) {
  return o.mn ? (uint32_t)ks * (2048u >> 4)
              : (uint32_t)(((ks >> 2) * o.R * 128 + (ks & 3) * 32) >> 4);
}

// One product D[M][N] (+)= A B^T, K = 16 per step, issued by one thread.
// The descriptors are formed once and stepped by constants, so the issuing
// thread spends its time on the MMAs rather than on descriptor arithmetic.
template <bool kLo>
struct Gemm {
  uint32_t d, id;
  uint64_t ah, bh, al, bl;
  const Operand *a, *b;
  bool accumulate;
  __device__ __forceinline__ Gemm(uint32_t d_, const Operand &a_,
                                  const Operand &b_, int M, int N,
                                  bool accumulate_)
      : d(d_),
        id(idesc_bf16(M, N, a_.mn, b_.mn)),
        ah(opdesc(a_, false)), bh(opdesc(b_, false)),
        al(kLo ? opdesc(a_, true) : 0), bl(kLo ? opdesc(b_, true) : 0),
        a(&a_), b(&b_), accumulate(accumulate_) {}
  // K step ks of the operands, accumulated onto D unless it is the first
  // step written (`first`) of a product that does not accumulate.
  __device__ __forceinline__ void step(int ks, bool first) const {
    const uint64_t ao = kstep16(*a, ks), bo = kstep16(*b, ks);
    mma_bf16(d, ah + ao, bh + bo, id, (accumulate || !first) ? 1u : 0u);
    if (kLo) {
      mma_bf16(d, ah + ao, bl + bo, id, 1u);
      mma_bf16(d, al + ao, bh + bo, id, 1u);
    }
  }
};

// The same with A in tensor memory (see mma_bf16_ta): the hi and lo parts
// of A start at TMEM addresses a and a_lo, and K step ks is 8 columns on.
template <bool kLo>
struct GemmT {
  uint32_t d, id, a, al;
  uint64_t bh, bl;
  const Operand *b;
  bool accumulate;
  __device__ __forceinline__ GemmT(uint32_t d_, uint32_t a_, uint32_t a_lo,
                                   const Operand &b_, int M, int N,
                                   bool accumulate_)
      : d(d_), id(idesc_bf16(M, N, 0, b_.mn)), a(a_), al(a_lo),
        bh(opdesc(b_, false)), bl(kLo ? opdesc(b_, true) : 0), b(&b_),
        accumulate(accumulate_) {}
  __device__ __forceinline__ void step(int ks, bool first) const {
    const uint64_t bo = kstep16(*b, ks);
    const uint32_t ao = 8u * (uint32_t)ks;
    mma_bf16_ta(d, a + ao, bh + bo, id, (accumulate || !first) ? 1u : 0u);
    if (kLo) {
      mma_bf16_ta(d, a + ao, bl + bo, id, 1u);
      mma_bf16_ta(d, al + ao, bh + bo, id, 1u);
    }
  }
};

template <int KSTEPS, class G>
__device__ __forceinline__ void gemm_steps(const G &g) {
#pragma unroll
  for (int ks = 0; ks < KSTEPS; ++ks) g.step(ks, ks == 0);
}

// Two independent products (different accumulators), their K steps
// interleaved so that one product's dependent chain runs while the other's
// waits.
template <int KSTEPS, class GX, class GY>
__device__ __forceinline__ void gemm2(const GX &x, const GY &y) {
#pragma unroll
  for (int ks = 0; ks < KSTEPS; ++ks) {
    x.step(ks, ks == 0);
    y.step(ks, ks == 0);
  }
}

__device__ __forceinline__ void cta_sync_tc() {
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
}

// Barrier among the kSimt threads of the SIMT warps only (named barrier 1);
// the issuing warp never takes part.
__device__ __forceinline__ void simt_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kSimt) : "memory");
}

// simt_sync that also returns whether `p` holds on every SIMT thread.
__device__ __forceinline__ bool simt_and(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, b;\n\t"
      "setp.ne.u32 a, %1, 0;\n\t"
      "bar.red.and.pred b, 1, %2, a;\n\t"
      "selp.u32 %0, 1, 0, b;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)p), "n"(kSimt)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar)
               : "memory");
}

// A SIMT thread's part of "operands ready": its shared-memory writes made
// visible to the tensor cores, its TMEM accesses ordered, then one arrival
// (the barrier completes after all kSimt arrivals).
__device__ __forceinline__ void signal_ready(uint32_t mbar) {
  fence_proxy_async();
  fence_before_sync();
  mbar_arrive(mbar);
}

// The one arrival of a phase, announcing `bytes` of bulk copies.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t mbar,
                                                      uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar),
               "r"(bytes)
               : "memory");
}

// Tensor copies of one box of a row tensor map (see rows_map): the 64
// token rows t0 .. t0+63 of head h of sequence b, 512 bytes each, to or from
// consecutive 512-byte rows of shared memory.  Rows past the sequence's end
// read as zeros and are not written.  The load counts its bytes (the whole
// box) against the mbarrier; the store joins this thread's bulk group.
__device__ __forceinline__ void tma_load_rows(uint32_t smem, const CUtensorMap *map,
                                              int h, int t0, int b, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(h), "r"(t0), "r"(b),
      "r"(mbar)
      : "memory");
}

__device__ __forceinline__ void tma_store_rows(const CUtensorMap *map, int h,
                                               int t0, int b, uint32_t smem) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group"
      " [%0, {%1, %2, %3, %4}], [%5];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(0), "r"(h), "r"(t0), "r"(b), "r"(smem)
      : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until all but the last `kPending` of this thread's committed groups
// of bulk stores have read their shared-memory source (which may then be
// overwritten), or (bulk_wait_all) until every one has completed.
template <int kPending>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kPending) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// fp32 scratch for the triangular solve: A and T, 64 x 64 each, rows of 64
// floats with the 16-byte groups of row r XOR-ed by (r & 7) so that eight
// consecutive rows at the same column hit different banks.
__device__ __forceinline__ int sidx(int r, int c) {
  return r * 64 + ((((c >> 2) ^ (r & 7)) << 2) | (c & 3));
}

__device__ __forceinline__ void put_row4(float *X, int r, int c, float4 v) {
  *reinterpret_cast<float4 *>(X + sidx(r, c)) = v;
}

__device__ __forceinline__ float4 get_row4(const float *X, int r, int c) {
  return *reinterpret_cast<const float4 *>(X + sidx(r, c));
}

// Element e (a compile-time index after unrolling) of a float4.
__device__ __forceinline__ float elem(const float4 &v, int e) {
  return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

// Y[r][c0..c0+3] = sum_{u0 <= u < n} X[xr][xc + u] * Z[zr + u][zc + c0 .. +3]
// over the fp32 scratch layout (u0, n multiples of 4); returns the four sums.
// (A compact loop: unrolled or software-pipelined forms of it measured
// slower here, the instruction footprint and the shared-memory loads
// counting for more than the load latency.)
__device__ __forceinline__ float4 row_times(const float *X, int xr, int xc,
                                            const float *Z, int zr, int zc,
                                            int n, int u0 = 0) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int u4 = u0; u4 < n; u4 += 4) {
    const float4 a = get_row4(X, xr, xc + u4);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float4 z = get_row4(Z, zr + u4 + e, zc);
      const float ae = elem(a, e);
      acc.x = fmaf(ae, z.x, acc.x);
      acc.y = fmaf(ae, z.y, acc.y);
      acc.z = fmaf(ae, z.z, acc.z);
      acc.w = fmaf(ae, z.w, acc.w);
    }
  }
  return acc;
}

// T = (I + A)^-1 for strictly lower-triangular A (64 x 64), by divide and
// conquer: invert the four 16 x 16 diagonal blocks, merge them into 32 x 32
// inverses, then into the 64 x 64 inverse, using
//   [[E1, 0], [A21, E2]]^-1 = [[E1^-1, 0], [-E2^-1 A21 E1^-1, E2^-1]].
// The kSimt SIMT threads.  Reads the lower triangle of Asc (its upper
// triangle is zero on entry and then holds the intermediate products);
// writes all of Tsc, zeros above the diagonal.  With kSide, warp 7 runs
// `side()` (work of its own that reads neither scratch) during the first
// step instead of taking part in it.
template <bool kSide, class Side>
__device__ __forceinline__ void tri_inverse(float *Asc, float *Tsc, int tid,
                                            Side &&side) {
  const int warp = tid >> 5, lane = tid & 31;
  if (warp < 2) {
    // 1. Diagonal blocks by forward substitution, one column per lane, in
    //    registers: warp w takes blocks 2w (lanes 0-15) and 2w + 1 (lanes
    //    16-31), lane its block's column jj.  p_t is the running sum of
    //    A[t][k] x_k over the x_k known so far; x_k is final once p_k has
    //    its k terms, and then enters the sums of the rows below it, so the
    //    serial chain per step is one subtraction and one FMA.  The sums
    //    run in order of k.
    const int hi = lane >> 4, jj = lane & 15;
    const int r0 = 32 * warp + 16 * hi;
    float x[16], p[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) p[t] = 0.f;
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
      float4 a[16];  // A[r0 + t][r0 + 4 k4 .. + 3] for the rows t below
#pragma unroll
      for (int t = 4 * k4 + 1; t < 16; ++t) a[t] = get_row4(Asc, r0 + t, r0 + 4 * k4);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int k = 4 * k4 + e;
        x[k] = (k == jj ? 1.f : 0.f) - p[k];
#pragma unroll
        for (int t = k + 1; t < 16; ++t) p[t] = fmaf(elem(a[t], e), x[k], p[t]);
      }
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) Tsc[sidx(r0 + t, r0 + jj)] = x[t];
  } else if (kSide && warp == kSimt / 32 - 1) {
    side();
  } else {
    // Meanwhile the other warps write the zeros above the block diagonal:
    // rows 0-15 of columns 16-31, rows 0-31 of 32-47, rows 0-47 of 48-63
    // (64 + 128 + 192 groups of four).
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int idx = tid - 64; idx < 384; idx += (kSide ? kSimt - 32 : kSimt) - 64) {
      const int b = idx < 64 ? 1 : idx < 192 ? 2 : 3;
      const int rel = idx - (b == 1 ? 0 : b == 2 ? 64 : 192);
      put_row4(Tsc, rel >> 2, 16 * b + 4 * (rel & 3), z);
    }
  }
  simt_sync();
  // 2. 16 -> 32: blocks (1,0) and (3,2).  Thread: block pair p, row r,
  //    columns 4 c4 .. 4 c4 + 3.  X = A_{i,i-1} E_{i-1} goes to the upper
  //    block (i-1, i) of the A scratch.
  if (tid < 128) {
    const int pr = tid >> 6, r = (tid >> 2) & 15, c4 = (tid & 3) * 4;
    const int i = 2 * pr + 1, j = i - 1;
    put_row4(Asc, 16 * j + r, 16 * i + c4,
             row_times(Asc, 16 * i + r, 16 * j, Tsc, 16 * j, 16 * j + c4, 16));
  }
  simt_sync();
  if (tid < 128) {
    const int pr = tid >> 6, r = (tid >> 2) & 15, c4 = (tid & 3) * 4;
    const int i = 2 * pr + 1, j = i - 1;
    // T_ij = -E_i X  (E_i = T block (i, i), X in A scratch block (j, i))
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u4 = 0; u4 < 16; u4 += 4) {
      const float4 e = get_row4(Tsc, 16 * i + r, 16 * i + u4);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 z = get_row4(Asc, 16 * j + u4 + q, 16 * i + c4);
        const float eq = elem(e, q);
        y.x = fmaf(eq, z.x, y.x);
        y.y = fmaf(eq, z.y, y.y);
        y.z = fmaf(eq, z.z, y.z);
        y.w = fmaf(eq, z.w, y.w);
      }
    }
    put_row4(Tsc, 16 * i + r, 16 * j + c4, make_float4(-y.x, -y.y, -y.z, -y.w));
  }
  simt_sync();
  // 3. 32 -> 64: X = A[32:64, 0:32] T[0:32, 0:32] goes to A scratch
  //    [0:32, 32:64]; then T[32:64, 0:32] = -T[32:64, 32:64] X.  Both T
  //    factors are exactly lower triangular, so the terms a warp skips are
  //    exact zeros: warp w takes columns 4w .. 4w+3 of X (rows = lanes) from
  //    k = 4w on, then rows 4w .. 4w+3 of the result (lanes: row 4w + lane/8,
  //    columns 4 (lane % 8)) up to k = 4w+3.  The sums keep their order.
  {
    const int c4 = 4 * warp;
    put_row4(Asc, lane, 32 + c4, row_times(Asc, 32 + lane, 0, Tsc, 0, c4, 32, c4));
  }
  simt_sync();
  {
    const int r = 4 * warp + (lane >> 3), c4 = (lane & 7) * 4;
    const float4 y = row_times(Tsc, 32 + r, 32, Asc, 0, 32 + c4, 4 * warp + 4);
    put_row4(Tsc, 32 + r, c4, make_float4(-y.x, -y.y, -y.z, -y.w));
  }
  simt_sync();
}

template <bool kLo>
__global__ void __launch_bounds__(kThreads, 1)
    gdn_chunk_kernel(float *__restrict__ S, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const float *__restrict__ g,
                     const float *__restrict__ beta,
                     const __grid_constant__ CUtensorMap tm_o,
                     float *__restrict__ o, int T, int kh, int vh, int rep) {
  // Where the gate warp makes the next chunk's gate vectors, while the
  // chunk still reads its own: warp 7 during the inverse's first step
  // (bf16), or warp 0 while the SIMT warps wait for the correction product
  // (split-bf16, where that wait is long; measured faster there than
  // during the inverse or under the chunk's last products).
  constexpr bool kGatesInInverse = !kLo;
  constexpr int kGateWarp = kGatesInInverse ? kSimt / 32 - 1 : 0;
  // gate-vector buffer of chunk c
  auto vbuf = [](int c) { return c & 1; };
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw_s = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t sb = (raw_s + 1023u) & ~1023u;
  unsigned char *gb = smem_raw + (sb - raw_s);
  // Gate vectors by chunk parity (see gates below): Gamma, gamma, w, beta,
  // and exp(Gamma_t - Gamma_s) = ea[t] eb[s] about the middle of the
  // chunk's range of Gamma, used when that range is at most 160 (fac != 0),
  // where every factor is a normal fp32 number.
  auto gvec = [&](int buf) {
    return reinterpret_cast<float *>(gb + (buf ? OFF_VEC1 : OFF_VEC));
  };
  volatile int *const fac2 = reinterpret_cast<volatile int *>(gb + OFF_BAR + 120);
  // mbarriers: products done (one commit each), operands ready (kSimt
  // arrivals each), and the final drain
  const uint32_t bar0 = sb + OFF_BAR;
  const uint32_t done_a = bar0, done_s = bar0 + 8, done_d = bar0 + 16,
                 done_4 = bar0 + 24;
  const uint32_t rdy_a = bar0 + 32, rdy_s = bar0 + 40, rdy_t = bar0 + 48,
                 rdy_d = bar0 + 56;
  const uint32_t drain = bar0 + 64;
  const uint32_t staged0 = bar0 + 72;  // K, Q rows of an even chunk in Ra
  const uint32_t v_free = bar0 + 80;   // the fp32 V rows in Rb are read
  const uint32_t vstaged = bar0 + 88;  // this chunk's fp32 V rows in region Rb
  const uint32_t staged1 = bar0 + 96;  // K, Q rows of an odd chunk in Rd
  const uint32_t kq_free = bar0 + 104; // a chunk's [K; Q] region is free again
  volatile uint32_t *slot = reinterpret_cast<volatile uint32_t *>(gb + OFF_SLOT);
  float *Asc = reinterpret_cast<float *>(gb + OFF_SCR);
  float *Tsc = Asc + 64 * 64;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3;      // TMEM lane quadrant of this warp
  const int half = (warp >> 2) & 1;  // which half of the columns this warp moves
  const int myrow = 32 * quad + lane;
  const uint32_t lane_base = (uint32_t)(32 * quad) << 16;

  const int head = blockIdx.x;
  const int b = head / vh, vi = head % vh, hh = vi / rep;
  const size_t head_off = (size_t)head * kD * kD;
  const int nchunks = (T + kC - 1) / kC;

  if (warp == 0) tmem_alloc(sb + OFF_SLOT, 512);
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(bar0 + 8 * i, 1);
    for (int i = 4; i < 8; ++i) mbar_init(bar0 + 8 * i, kSimt);
    mbar_init(drain, 1);
    mbar_init(staged0, 1);
    mbar_init(staged1, 1);
    mbar_init(kq_free, 1);
    mbar_init(v_free, 1);
    mbar_init(vstaged, 1);
  }
  cta_sync_tc();
  const uint32_t tmem = *slot;

  if (warp == kLoader) {
    // ------------------------------------------------ the copying warp
    // K and Q rows of chunk c, fp32, into its region (Ra for even c, Rd for
    // odd c) once chunk c-2's products have finished reading that region:
    // a chunk ahead of use.  Then its fp32 V rows into region Rb once the
    // SIMT warps have read chunk c-1's.  One tensor copy of 64
    // rows each; rows past T arrive as zeros.
    int issued[2] = {-1, -1}, v_issued = -1;
    for (int c = 0; c < nchunks; ++c) {
      if (c >= 2 && !mbar_wait(kq_free, (uint32_t)((c - 2) & 1), kWaitLimit)) break;
      const uint32_t st = (c & 1) ? staged1 : staged0;
      if (lane == 0) {
        mbar_arrive_expect_tx(st, 2u * kC * 512u);
        tma_load_rows(sb + kq_region(c), &tm_k, hh, c * kC, b, st);
        tma_load_rows(sb + kq_region(c) + kC * 512, &tm_q, hh, c * kC, b, st);
      }
      __syncwarp();
      issued[c & 1] = c;
      if (c > 0 && !mbar_wait(v_free, (uint32_t)((c - 1) & 1), kWaitLimit)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(vstaged, kC * 512u);
        tma_load_rows(sb + OFF_V, &tm_v, vi, c * kC, b, vstaged);
      }
      __syncwarp();
      v_issued = c;
    }
    // nothing may still be copying into shared memory when the CTA ends
    for (int j = 0; j < 2; ++j)
      if (issued[j] >= 0)
        mbar_wait(j ? staged1 : staged0, (uint32_t)((issued[j] >> 1) & 1), kWaitLimit);
    if (v_issued >= 0) mbar_wait(vstaged, (uint32_t)(v_issued & 1), kWaitLimit);
  } else if (warp == kIssuer) {
    // ------------------------------------------------ the issuing warp
    // One thread issues every product of every chunk as soon as the SIMT
    // warps report its operands ready; tcgen05.mma issue waits while the
    // tensor pipe is busy, and here that wait holds up no SIMT work.
    if (lane == 0) {
      const Operand opTB2{sb + OFF_TB2, 64, 64, false};   // MMA-ud B
      const Operand opP{sb + OFF_P, 64, 64, false};       // MMA-3 B
      uint32_t ph = 0;
      for (int c = 0; c < nchunks; ++c) {
        const uint32_t kq = sb + kq_region(c);
        const Operand opKQ{kq, 128, 128, false};   // MMA-a A; MMA-s B ([K; Q])
        const Operand opKb{kq, 128, 128, false};   // MMA-a B (K: rows 0-63)
        const Operand opKnB{kq, 128, 128, true};   // MMA-4 B (K rows)
        if (!mbar_wait(rdy_a, ph, kWaitLimit)) break;
        fence_after_sync();
        {
          // [K;Q] K^T as two half-K products in two accumulators (T_U is
          // free until MMA-ud); the A/P build adds them
          const Gemm<kLo> lo_(tmem + T_GH, opKQ, opKb, 128, kC, false);
          const Gemm<kLo> hi_(tmem + T_U, opKQ, opKb, 128, kC, false);
#pragma unroll
          for (int ks = 0; ks < kD / 32; ++ks) {
            lo_.step(ks, ks == 0);
            hi_.step(ks + kD / 32, ks == 0);
          }
        }
        commit(done_a);
        if (!mbar_wait(rdy_s, ph, kWaitLimit)) break;
        fence_after_sync();
        gemm_steps<kD / 16>(GemmT<kLo>(tmem + T_BUF, tmem + T_AOP, tmem + T_AOP + 64,
                                       opKQ, 128, 2 * kC, false));
        commit(done_s);
        if (!mbar_wait(rdy_t, ph, kWaitLimit)) break;
        fence_after_sync();
        gemm_steps<kC / 16>(GemmT<kLo>(tmem + T_U, tmem + T_AOP, tmem + T_AOP + 32,
                                       opTB2, 128, kC, false));
        commit(done_d);
        if (!mbar_wait(rdy_d, ph, kWaitLimit)) break;
        fence_after_sync();
        gemm2<kC / 16>(GemmT<kLo>(tmem + T_BUF, tmem + T_AOP, tmem + T_AOP + 32, opP,
                                  128, kC, false),
                       GemmT<kLo>(tmem + T_SACC, tmem + T_AOP + 64, tmem + T_AOP + 96,
                                  opKnB, 128, kD, true));
        commit(done_4);
        ph ^= 1u;
      }
      commit(drain);  // arrives once every product issued above is done
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ the SIMT warps
    const uint32_t tl = tmem + lane_base;

    // On the gate warp, the next chunk's g and beta of tokens lane and
    // lane + 32 in registers.  (K, Q and V come by tensor copy.)
    float pg[2], pb[2];
    auto prefetch = [&](int c) {
      const int t0 = c * kC;
      const int n = min(kC, T - t0);
      const size_t v_base = ((size_t)b * T + t0) * vh + vi;
      if (warp == kGateWarp) {
        pg[0] = lane < n ? __ldg(g + v_base + (size_t)lane * vh) : 0.f;
        pg[1] = lane + 32 < n ? __ldg(g + v_base + (size_t)(lane + 32) * vh) : 0.f;
        pb[0] = lane < n ? __ldg(beta + v_base + (size_t)lane * vh) : 0.f;
        pb[1] = lane + 32 < n ? __ldg(beta + v_base + (size_t)(lane + 32) * vh) : 0.f;
      }
    };
    if (warp == kGateWarp) prefetch(0);

    // State in: S[dk][dv] -> TMEM lane dv, column dk.
    {
      const float *Sh = S + head_off;
      for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 16) {
        float r[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) r[j] = __ldg(Sh + (size_t)(c0 + j) * kD + myrow);
        tmem_st16(tl + T_SACC + c0, r);
      }
    }

    // o for chunk cc = diag(gamma) (Q S)^T + (P Delta)^T, read from TMEM
    // into the o tile ([t][dv] rows of 512 bytes, the layout of o), then
    // written out by two tensor stores (store_o) after a SIMT barrier, so
    // the global stores leave the SIMT warps' path.
    float *otile = reinterpret_cast<float *>(gb + OFF_OT);
    auto emit_o = [&](int cc) {
      const float *gm = gvec(cc & 1) + 64;  // gamma of chunk cc
      const uint32_t pdq = T_BUF;
      for (int c0 = half * 32; c0 < half * 32 + 32; c0 += 16) {
        float r[16], pd[16];
        tmem_ld16(tl + pdq + 64 + c0, r);
        tmem_ld16(tl + pdq + c0, pd);
#pragma unroll
        for (int j4 = 0; j4 < 16; j4 += 4) {
          const float4 g4 = *reinterpret_cast<const float4 *>(gm + c0 + j4);
          otile[(c0 + j4) * kD + myrow] = fmaf(g4.x, r[j4], pd[j4]);
          otile[(c0 + j4 + 1) * kD + myrow] = fmaf(g4.y, r[j4 + 1], pd[j4 + 1]);
          otile[(c0 + j4 + 2) * kD + myrow] = fmaf(g4.z, r[j4 + 2], pd[j4 + 2]);
          otile[(c0 + j4 + 3) * kD + myrow] = fmaf(g4.w, r[j4 + 3], pd[j4 + 3]);
        }
      }
      fence_proxy_async();  // the tile is read by the copy engine
    };
    // Thread 0, after the barrier that follows emit_o(cc): the tile's two
    // halves of 32 rows by one tensor store each, in two commit groups, so
    // the first half (the A scratch's region) is free once its own store has
    // read it.  Rows past T are not written; a half that starts past T is
    // not stored (only the last chunk's can).
    auto store_o = [&](int cc) {
      tma_store_rows(&tm_o, vi, cc * kC, b, sb + OFF_OT);
      bulk_commit();
      if (cc * kC + kC / 2 < T) {
        tma_store_rows(&tm_o, vi, cc * kC + kC / 2, b, sb + OFF_OT + kC / 2 * kD * 4);
        bulk_commit();
      }
    };

    // Gate vectors of chunk cc from the prefetched g, beta (the gate warp):
    // the cumulative log-decay Gamma, gamma, w, beta, the factors ea, eb,
    // into buffer cc & 1.  Run for chunk c + 1 during chunk c (see
    // kGatesInInverse), before a SIMT barrier that makes them visible; the
    // buffer's previous contents (chunk c - 1) were last read by that
    // chunk's output, at the top of chunk c.
    auto gates = [&](int cc) {
      float *Gam = gvec(vbuf(cc));
      float *gam = Gam + 64, *wv = Gam + 128, *bet = Gam + 192;
      float *ea = Gam + 384, *eb = Gam + 448;
      bet[lane] = pb[0];
      bet[lane + 32] = pb[1];
      float sa = pg[0], sc = pg[1];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float ya = __shfl_up_sync(0xffffffffu, sa, off);
        const float yc = __shfl_up_sync(0xffffffffu, sc, off);
        if (lane >= off) {
          sa += ya;
          sc += yc;
        }
      }
      sc += __shfl_sync(0xffffffffu, sa, 31);
      const float last = __shfl_sync(0xffffffffu, sc, 31);
      Gam[lane] = sa;
      Gam[lane + 32] = sc;
      gam[lane] = expf(sa);
      gam[lane + 32] = expf(sc);
      wv[lane] = expf(last - sa);
      wv[lane + 32] = expf(last - sc);
      float gmax = fmaxf(sa, sc), gmin = fminf(sa, sc);
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, off));
        gmin = fminf(gmin, __shfl_xor_sync(0xffffffffu, gmin, off));
      }
      const float ref = 0.5f * (gmax + gmin);
      ea[lane] = expf(sa - ref);
      ea[lane + 32] = expf(sc - ref);
      eb[lane] = expf(ref - sa);
      eb[lane + 32] = expf(ref - sc);
      if (lane == 0) fac2[vbuf(cc)] = (gmax - gmin <= 160.f) ? 1 : 0;
    };
    if (warp == kGateWarp) gates(0);
    // [K; Q] operand of chunk cc, in place in its region: this thread's
    // fp32 rows (tid >> 4) + 16 i, columns (tid & 15) * 8 .. + 7, are read
    // into registers, then, after a barrier, written back as bf16 operand
    // rows.  Lanes 4-7 of each quarter warp read their two 16-byte halves
    // in the other order, so each of the two loads covers all eight 16-byte
    // bank groups of the quarter warp once.  False if the rows never came.
    auto kq_operand = [&](int cc) -> bool {
      const uint32_t st = (cc & 1) ? staged1 : staged0;
      if (!simt_and(mbar_wait(st, (uint32_t)((cc >> 1) & 1), kWaitLimit))) return false;
      const float *stage = reinterpret_cast<const float *>(gb + kq_region(cc));
      const int swap = (tid >> 2) & 1, c0 = (tid & 15) * 8;
      float x[8][8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int row = (tid >> 4) + 16 * i;
        const float4 ya = *reinterpret_cast<const float4 *>(stage + row * 128 + c0 + 4 * swap);
        const float4 yb = *reinterpret_cast<const float4 *>(stage + row * 128 + c0 + 4 - 4 * swap);
        const float4 x0 = swap ? yb : ya, x1 = swap ? ya : yb;
        x[i][0] = x0.x; x[i][1] = x0.y; x[i][2] = x0.z; x[i][3] = x0.w;
        x[i][4] = x1.x; x[i][5] = x1.y; x[i][6] = x1.z; x[i][7] = x1.w;
      }
      simt_sync();
#pragma unroll
      for (int i = 0; i < 8; ++i)
        put8<kLo>(gb, kq_region(cc), 128, 128, (tid >> 4) + 16 * i, c0, x[i]);
      return true;
    };
    uint32_t parity = 0;
    bool failed = !kq_operand(0);
    if (!failed) signal_ready(rdy_a);  // -> MMA-a of chunk 0
    for (int c = 0; !failed && c < nchunks; ++c) {
      // ---------------------------------------------------- phase 0: inputs
      // This chunk's [K; Q] operand was made, and MMA-a released, during
      // the previous chunk's last products, and its gates during the
      // previous chunk's inverse (both before the loop for chunk 0).
      const float *Gam = gvec(vbuf(c));
      const float *gam = Gam + 64, *wv = Gam + 128, *bet = Gam + 192;
      const float *ea = Gam + 384, *eb = Gam + 448;
      if (warp == kGateWarp && c + 1 < nchunks) prefetch(c + 1);  // for gates(c + 1)
      if (c > 0) emit_o(c - 1);  // the previous chunk's output, into the o tile
      simt_sync();  // the o tile is written
      if (c > 0 && tid == 0) store_o(c - 1);

      // ------------- phase 1: S^T operand (lane dv, K = dk) in TMEM; the
      // accumulator is then decayed in place, S^T *= gamma_63, ready for
      // MMA-4 (nothing reads it in between: MMA-s reads the operand)
      {
        const float gC = gam[kC - 1];
        for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 16) {
          float r[16];
          tmem_ld16(tl + T_SACC + c0, r);
          put16_tmem<kLo>(tl + T_AOP, tl + T_AOP + 64, c0, r);
#pragma unroll
          for (int j = 0; j < 16; ++j) r[j] *= gC;
          tmem_st16(tl + T_SACC + c0, r);  // waits for this thread's stores
        }
      }
      signal_ready(rdy_s);  // -> MMA-s: [Y | (Q S)^T] = S^T [K; Q]^T
      // the o tile's first half is reused by the A scratch (both halves
      // were stored: chunk c - 1 is a full chunk)
      if (c > 0 && tid == 0) bulk_wait_read<1>();
      if (!simt_and(mbar_wait(done_a, parity, kWaitLimit))) { failed = true; break; }
      fence_after_sync();

      // ----------------- phase 2: A and P, T = (I + A)^-1, T diag operands
      const bool factored = fac2[vbuf(c)] != 0;
      if (quad < 2) {  // lanes 0-63 hold G rows t
        const int t = myrow;
        const float bt = bet[t], Gt = Gam[t], bea = bt * ea[t];
        for (int c0 = half * 32; c0 < half * 32 + 32; c0 += 16) {
          float r[16], r2[16];
          tmem_ld16(tl + T_GH + c0, r);
          tmem_ld16(tl + T_U + c0, r2);
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] += r2[e];
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            float4 a4;
            float *a = &a4.x;
            if (factored) {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int s = c0 + 4 * j4 + e;
                a[e] = s < t ? bea * eb[s] * r[4 * j4 + e] : 0.f;
              }
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int s = c0 + 4 * j4 + e;
                a[e] = s < t ? bt * expf(Gt - Gam[s]) * r[4 * j4 + e] : 0.f;
              }
            }
            *reinterpret_cast<float4 *>(Asc + sidx(t, c0 + 4 * j4)) = a4;
          }
        }
      } else {  // lanes 64-127 hold H rows t: P straight to its operand
        const int t = myrow - kC;
        const float Gt = Gam[t], et = ea[t];
        for (int c0 = half * 32; c0 < half * 32 + 32; c0 += 16) {
          float r[16], r2[16];
          tmem_ld16(tl + T_GH + c0, r);
          tmem_ld16(tl + T_U + c0, r2);
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] += r2[e];
          if (factored) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int s = c0 + e;
              r[e] = s <= t ? et * eb[s] * r[e] : 0.f;
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int s = c0 + e;
              r[e] = s <= t ? expf(Gt - Gam[s]) * r[e] : 0.f;
            }
          }
          put8<kLo>(gb, OFF_P, kC, kC, t, c0, r);
          put8<kLo>(gb, OFF_P, kC, kC, t, c0 + 8, r + 8);
        }
      }
      // The A operand of the correction product in TMEM (lane dv, K = s):
      // V^T - Y diag(gamma), since Delta^T = U^T - (W S)^T
      // = V^T (T diag(beta))^T - Y (T diag(beta gamma))^T
      // = (V^T - Y diag(gamma)) (T diag(beta))^T.  V comes from its fp32
      // rows in region Rb (row s, this lane's column), Y from MMA-s.
      // (The wait is also the barrier between the A build and the inverse,
      // and, on thread 0, for the o tile's second half, which the inverse's
      // T scratch reuses.)
      if (c > 0 && tid == 0) bulk_wait_read<0>();
      if (!simt_and(mbar_wait(done_s, parity, kWaitLimit) &&
                    mbar_wait(vstaged, parity, kWaitLimit))) { failed = true; break; }
      fence_after_sync();
      {
        const float *vst = reinterpret_cast<const float *>(gb + OFF_V);
        for (int c0 = half * 32; c0 < half * 32 + 32; c0 += 16) {
          float r[16];
          tmem_ld16(tl + T_BUF + c0, r);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            r[e] = fmaf(-r[e], gam[c0 + e], vst[(c0 + e) * kD + myrow]);
          put16_tmem<kLo>(tl + T_AOP, tl + T_AOP + 32, c0, r);
        }
      }
      if constexpr (kGatesInInverse)
        tri_inverse<true>(Asc, Tsc, tid, [&] {
          if (c + 1 < nchunks) gates(c + 1);
        });
      else
        tri_inverse<false>(Asc, Tsc, tid, [] {});
      // (its barriers also follow every read of the V rows above)
      if (tid == 0) mbar_arrive(v_free);

      // T diag(beta), the B operand, over the A scratch (the inverse has
      // finished with it); each thread takes one row-half of T: row
      // t = tid >> 2, 16 columns
      const int t_row = tid >> 2, cq = (tid & 3) * 16;
      float tr[16];
#pragma unroll
      for (int e4 = 0; e4 < 16; e4 += 4) {
        const float4 v4 = *reinterpret_cast<const float4 *>(Tsc + sidx(t_row, cq + e4));
        tr[e4] = v4.x;
        tr[e4 + 1] = v4.y;
        tr[e4 + 2] = v4.z;
        tr[e4 + 3] = v4.w;
      }
#pragma unroll
      for (int h8 = 0; h8 < 2; ++h8) {
        float x2[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x2[e] = tr[8 * h8 + e] * bet[cq + 8 * h8 + e];
        put8<kLo>(gb, OFF_TB2, kC, kC, t_row, cq + 8 * h8, x2);
      }
      tmem_wait_st();
      signal_ready(rdy_t);  // -> MMA-ud: Delta^T = (V^T - Y diag(gamma)) (T diag(beta))^T
      if (!kGatesInInverse && warp == kGateWarp && c + 1 < nchunks) gates(c + 1);
      if (!simt_and(mbar_wait(done_d, parity, kWaitLimit))) { failed = true; break; }
      fence_after_sync();

      // ------------- phase 4: Delta^T, Delta^T diag(w) operands in TMEM
      for (int c0 = half * 32; c0 < half * 32 + 32; c0 += 16) {
        float u[16];
        tmem_ld16(tl + T_U + c0, u);
        put16_tmem<kLo>(tl + T_AOP, tl + T_AOP + 32, c0, u);
#pragma unroll
        for (int e = 0; e < 16; ++e) u[e] *= wv[c0 + e];
        put16_tmem<kLo>(tl + T_AOP + 64, tl + T_AOP + 96, c0, u);
      }
      tmem_wait_st();
      signal_ready(rdy_d);  // -> MMA-3: (P Delta)^T;  MMA-4: S^T += ...
      if (c + 1 < nchunks) {
        // Under MMA-3 and MMA-4: the next chunk's [K; Q] operand (in the
        // other region); then MMA-a of the next chunk is released (it queues
        // behind this chunk's products).
        if (!kq_operand(c + 1)) { failed = true; break; }
        signal_ready(rdy_a);
      }
      if (!simt_and(mbar_wait(done_4, parity, kWaitLimit))) { failed = true; break; }
      fence_after_sync();
      // this chunk's [K; Q] region may take the rows of chunk c + 2
      if (tid == 0) mbar_arrive(kq_free);
      parity ^= 1u;
    }

    if (!failed) {
      emit_o(nchunks - 1);
      simt_sync();
      if (tid == 0) store_o(nchunks - 1);
      float *Sh = S + head_off;
      for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 16) {
        float r[16];
        tmem_ld16(tl + T_SACC + c0, r);
#pragma unroll
        for (int j = 0; j < 16; ++j) Sh[(size_t)(c0 + j) * kD + myrow] = r[j];
      }
    } else {
      // a wait ran out: the head's state and every o row of the head become
      // NaN (after the tensor stores already issued have landed), so the
      // failure shows in the results as well as in the counter
      if (tid == 0) {
        atomicAdd(&g_prefill_timeouts, 1u);
        bulk_wait_all();
      }
      simt_sync();
      const float nan = __int_as_float(0x7fffffff);
      float *Sh = S + head_off;
      for (int e = tid; e < kD * kD; e += kSimt) Sh[e] = nan;
      for (size_t e = tid; e < (size_t)T * kD; e += kSimt) {
        const size_t t = e / kD;
        o[(((size_t)b * T + t) * vh + vi) * kD + (e - t * kD)] = nan;
      }
    }
    if (tid == 0) bulk_wait_all();  // no store of o outlives the CTA
  }
  // every product issued has finished (bounded: after a timeout the issuer
  // stops early and its drain commit still arrives)
  mbar_wait(drain, 0, kWaitLimit);
  cta_sync_tc();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

size_t prefill_workspace_bytes(int, int, int, int, int, int) { return 0; }

namespace {

// cuTensorMapEncodeTiled, from the driver through the runtime (the library
// does not link the driver library itself); null if it is unavailable.
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tensor map over a [B][T][heads][128] fp32 array (q, k, v or o) as a 4-d
// tensor {128, heads, T, B}; one box is `rows` token rows of one head of one
// sequence.  Rows past T are outside the tensor: zeros when loaded, skipped
// when stored.
cudaError_t rows_map(CUtensorMap *map, const float *base, int heads, int T,
                     int B, int rows) {
  const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_tiled();
  if (fn == nullptr) return cudaErrorNotSupported;
  const cuuint64_t row = (cuuint64_t)kD * sizeof(float);
  const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)heads, (cuuint64_t)T,
                              (cuuint64_t)B};
  const cuuint64_t strides[3] = {row, row * (cuuint64_t)heads,
                                 row * (cuuint64_t)heads * (cuuint64_t)T};
  const cuuint32_t box[4] = {(cuuint32_t)kD, 1, (cuuint32_t)rows, 1};
  const cuuint32_t step[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                        const_cast<float *>(base), dims, strides, box, step,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill_chunked(float *S, const float *q, const float *k,
                                   const float *v, const float *g,
                                   const float *beta, float *o, int B, int kh,
                                   int vh, int T, int precision, void *,
                                   cudaStream_t stream) {
  const size_t nheads = (size_t)B * vh;
  if (nheads == 0) return cudaSuccess;
  if (nheads > 0x7fffffffull) return cudaErrorInvalidConfiguration;
  CUtensorMap tm_q, tm_k, tm_v, tm_o;
  cudaError_t e;
  if ((e = rows_map(&tm_q, q, kh, T, B, kC)) != cudaSuccess) return e;
  if ((e = rows_map(&tm_k, k, kh, T, B, kC)) != cudaSuccess) return e;
  if ((e = rows_map(&tm_v, v, vh, T, B, kC)) != cudaSuccess) return e;
  if ((e = rows_map(&tm_o, o, vh, T, B, kC / 2)) != cudaSuccess) return e;
  if (precision == 1) {
    e = cudaFuncSetAttribute(gdn_chunk_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    gdn_chunk_kernel<true><<<(unsigned)nheads, kThreads, kSmemAlloc, stream>>>(
        S, tm_q, tm_k, tm_v, g, beta, tm_o, o, T, kh, vh, vh / kh);
  } else {
    e = cudaFuncSetAttribute(gdn_chunk_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    gdn_chunk_kernel<false><<<(unsigned)nheads, kThreads, kSmemAlloc, stream>>>(
        S, tm_q, tm_k, tm_v, g, beta, tm_o, o, T, kh, vh, vh / kh);
  }
  return cudaGetLastError();
}

cudaError_t prefill_timeouts(unsigned int *count) {
  return cudaMemcpyFromSymbol(count, g_prefill_timeouts, sizeof(unsigned int));
}

}  // namespace gdn
