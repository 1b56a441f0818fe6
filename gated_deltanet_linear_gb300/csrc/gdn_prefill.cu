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
// column per key row dk) in tensor memory for the whole sequence.  Per
// chunk (D = M x N accumulator in TMEM, lanes = M):
//   MMA-a  G,H  [t'][s]  = [K; Q] K^T                       (A, B K-major)
//   SIMT   A from G; T = (I + A)^-1, blocked 16 x 16, fp32
//   MMA-w  W^T  [dk][t]  = K^T (T diag(beta gamma))^T       (A = K, MN-major)
//   MMA-u  U^T  [dv][t]  = V^T (T diag(beta))^T             (A = V, MN-major)
//   MMA-1  Delta^T = U^T - S^T W^T (negated A, accumulated onto U^T);
//          (Q S)^T [dv][t] = S^T Q^T                        (B = W^T, MN-major)
//   SIMT   Delta^T also scaled by w;  S^T *= gamma_63;  P (built with A)
//   MMA-3  (P Delta)^T = Delta^T P^T
//   MMA-4  S^T += (Delta^T diag(w)) K                        (B = K, MN-major)
//   SIMT   O^T = diag(gamma) (Q S)^T + (P Delta)^T  -> o, emitted while the
//          next chunk's first product runs
// Every operand a thread writes is a row it owns (a row of an input, or a
// TMEM lane of an earlier result), stored 8 elements at a time; transposes
// happen in the MMA descriptors (MN-major operands), never in memory.  The
// next chunk's K, Q, V rows and gates are loaded into registers while the
// current chunk's last products run.
//
// Precision.  Operands are bf16 in shared memory:
//   split-bf16 ("BF16X3"): x = hi + lo with hi = bf16(x), lo = bf16(x - hi);
//     a product is hi*hi + hi*lo + lo*hi, three MMAs with fp32 accumulation
//     (about 16 significant bits per operand; ~1e-5 relative error);
//   plain bf16: hi only, one MMA per product (~1e-2 relative error).
// The triangular solve, the gating exponentials and every accumulation are
// fp32.

#include <cuda_bf16.h>

#include "gdn_internal.cuh"
#include "gdn_tc.cuh"

namespace gdn {

__device__ unsigned int g_prefill_timeouts = 0;

namespace {

using namespace tc;

constexpr int kC = 64;       // chunk length
constexpr int kD = kDim;     // 128
constexpr int kThreads = 256;

// Operand tiles: R rows x C bf16 columns, 128-byte-swizzled blocks of 64
// columns (see gdn_tc.cuh), hi tile followed by lo tile (R * C * 2 bytes
// each).  Regions (byte offsets from a 1024-aligned base) are reused by
// phase:
//   Ra 64 KB: [K; Q] (128 x 128), the whole chunk
//   Rb 32 KB: V (64 x 128)            -> Delta^T (128 x 64)
//   Rc 32 KB: A, T scratch (fp32)     -> T diag(bg), T diag(b) (64 x 64 each)
//                                     -> W^T (128 x 64) -> Delta^T diag(w)
//   Rd 64 KB: S^T (128 x 128)         -> P (64 x 64)
constexpr uint32_t RA = 0, RB = 65536, RC = 98304, RD = 131072;
constexpr uint32_t OFF_KQ = RA;             // 128 x 128
constexpr uint32_t OFF_V = RB;              // 64 x 128
constexpr uint32_t OFF_DT = RB;             // 128 x 64 (after MMA-u)
constexpr uint32_t OFF_SCR = RC;            // fp32 A [64][64] + T [64][64]
constexpr uint32_t OFF_TB = RC;             // 64 x 64: T diag(beta gamma)
constexpr uint32_t OFF_TB2 = RC + 16384;    // 64 x 64: T diag(beta)
constexpr uint32_t OFF_WT = RC;             // 128 x 64 (after MMA-w/u)
constexpr uint32_t OFF_DTW = RC;            // 128 x 64 (after MMA-1)
constexpr uint32_t OFF_ST = RD;             // 128 x 128
constexpr uint32_t OFF_P = RD;              // 64 x 64 (after MMA-1)
constexpr uint32_t OFF_VEC = RD + 65536;    // Gamma, gamma, w, beta, gamma x 2
constexpr uint32_t OFF_BAR = OFF_VEC + 2048;
constexpr uint32_t kSmemUsed = OFF_BAR + 64;
constexpr uint32_t kSmemAlloc = kSmemUsed + 1024;  // room to align the base

// TMEM columns (512 allocated).
constexpr uint32_t T_SACC = 0;    // S^T: lanes dv, 128 columns dk
constexpr uint32_t T_GH = 128;    // G (lanes 0-63), H then P (lanes 64-127): 64 columns
constexpr uint32_t T_W = 192;     // W^T: lanes dk, columns t
constexpr uint32_t T_U = 256;     // U^T, then Delta^T = U^T - (W S)^T: lanes dv
constexpr uint32_t T_QS = 384;    // (Q S)^T: lanes dv, columns t
constexpr uint32_t T_PD = 448;    // (P Delta)^T: lanes dv, columns t

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

// D[M][N] (+)= A B^T over K = 16 * ksteps, issued by one thread.
template <bool kLo>
__device__ __forceinline__ void gemm(uint32_t d, const Operand &a,
                                     const Operand &b, int M, int N,
                                     int ksteps, bool accumulate,
                                     bool negate_a = false) {
  const uint32_t id = idesc_bf16(M, N, a.mn, b.mn) | (negate_a ? (1u << 13) : 0u);
  const uint32_t a_lo = a.base + (uint32_t)(a.R * a.C * 2);
  const uint32_t b_lo = b.base + (uint32_t)(b.R * b.C * 2);
  for (int ks = 0; ks < ksteps; ++ks) {
    const uint64_t ah = a.mn ? mnmajor(a.base, a.R, ks) : kmajor(a.base, a.R, ks);
    const uint64_t bh = b.mn ? mnmajor(b.base, b.R, ks) : kmajor(b.base, b.R, ks);
    mma_bf16(d, ah, bh, id, (accumulate || ks > 0) ? 1u : 0u);
    if (kLo) {
      const uint64_t bl = b.mn ? mnmajor(b_lo, b.R, ks) : kmajor(b_lo, b.R, ks);
      const uint64_t al = a.mn ? mnmajor(a_lo, a.R, ks) : kmajor(a_lo, a.R, ks);
      mma_bf16(d, ah, bl, id, 1u);
      mma_bf16(d, al, bh, id, 1u);
    }
  }
}

__device__ __forceinline__ void cta_sync_tc() {
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
}

// fp32 scratch for the triangular solve: A and T, 64 x 64 each, rows of 64
// floats with the 16-byte groups of row r XOR-ed by (r & 7) so that eight
// consecutive rows at the same column hit different banks.
__device__ __forceinline__ int sidx(int r, int c) {
  return r * 64 + ((((c >> 2) ^ (r & 7)) << 2) | (c & 3));
}

// Y[r][c0..c0+3] = sum_{u < n} X[xr][xc + u] * Z[zr + u][zc + c0 .. +3] over
// the fp32 scratch layout; returns the four sums.
__device__ __forceinline__ float4 row_times(const float *X, int xr, int xc,
                                            const float *Z, int zr, int zc,
                                            int n) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int u4 = 0; u4 < n; u4 += 4) {
    const float4 a = *reinterpret_cast<const float4 *>(X + sidx(xr, xc + u4));
    const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float4 z = *reinterpret_cast<const float4 *>(Z + sidx(zr + u4 + e, zc));
      acc.x = fmaf(av[e], z.x, acc.x);
      acc.y = fmaf(av[e], z.y, acc.y);
      acc.z = fmaf(av[e], z.z, acc.z);
      acc.w = fmaf(av[e], z.w, acc.w);
    }
  }
  return acc;
}

__device__ __forceinline__ void put_row4(float *X, int r, int c, float4 v) {
  *reinterpret_cast<float4 *>(X + sidx(r, c)) = v;
}

// T = (I + A)^-1 for strictly lower-triangular A (64 x 64), by divide and
// conquer: invert the four 16 x 16 diagonal blocks, merge them into 32 x 32
// inverses, then into the 64 x 64 inverse, using
//   [[E1, 0], [A21, E2]]^-1 = [[E1^-1, 0], [-E2^-1 A21 E1^-1, E2^-1]].
// All 256 threads.  Reads the lower triangle of Asc; its upper triangle
// (zero, never read as A) holds the intermediate products.  Writes Tsc.
__device__ __forceinline__ void tri_inverse(float *Asc, float *Tsc, int tid) {
  // 1. Diagonal blocks by forward substitution: column j of block i on 4
  //    lanes, rows split by r mod 4.
  {
    const int col = tid >> 2;          // 0..63: block i = col / 16
    const int q4 = tid & 3;
    const int blk = col >> 4, jj = col & 15, r0 = blk * 16;
    float x[4] = {0.f, 0.f, 0.f, 0.f};  // rows r0 + q4 + 4i
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        part = fmaf(Asc[sidx(r0 + t, r0 + q4 + 4 * i)], x[i], part);
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      const float xt = (t == jj ? 1.f : 0.f) - part;
      if ((t & 3) == q4) x[t >> 2] = xt;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) Tsc[sidx(r0 + q4 + 4 * i, r0 + jj)] = x[i];
    // zero the strictly-upper part of this column
    for (int r = q4; r < r0; r += 4) Tsc[sidx(r, r0 + jj)] = 0.f;
  }
  __syncthreads();
  // 2. 16 -> 32: blocks (1,0) and (3,2).  Thread: block pair p, row r,
  //    columns 4 c4 .. 4 c4 + 3.  X = A_{i,i-1} E_{i-1} goes to the upper
  //    block (i-1, i) of the A scratch.
  if (tid < 128) {
    const int pr = tid >> 6, r = (tid >> 2) & 15, c4 = (tid & 3) * 4;
    const int i = 2 * pr + 1, j = i - 1;
    put_row4(Asc, 16 * j + r, 16 * i + c4,
             row_times(Asc, 16 * i + r, 16 * j, Tsc, 16 * j, 16 * j + c4, 16));
  }
  __syncthreads();
  if (tid < 128) {
    const int pr = tid >> 6, r = (tid >> 2) & 15, c4 = (tid & 3) * 4;
    const int i = 2 * pr + 1, j = i - 1;
    // T_ij = -E_i X  (E_i = T block (i, i), X in A scratch block (j, i))
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u4 = 0; u4 < 16; u4 += 4) {
      const float4 e = *reinterpret_cast<const float4 *>(Tsc + sidx(16 * i + r, 16 * i + u4));
      const float ev[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 z = *reinterpret_cast<const float4 *>(Asc + sidx(16 * j + u4 + q, 16 * i + c4));
        y.x = fmaf(ev[q], z.x, y.x);
        y.y = fmaf(ev[q], z.y, y.y);
        y.z = fmaf(ev[q], z.z, y.z);
        y.w = fmaf(ev[q], z.w, y.w);
      }
    }
    put_row4(Tsc, 16 * i + r, 16 * j + c4, make_float4(-y.x, -y.y, -y.z, -y.w));
  }
  __syncthreads();
  // 3. 32 -> 64: X = A[32:64, 0:32] T[0:32, 0:32] goes to A scratch
  //    [0:32, 32:64]; then T[32:64, 0:32] = -T[32:64, 32:64] X.
  {
    const int r = tid >> 3, c4 = (tid & 7) * 4;
    put_row4(Asc, r, 32 + c4, row_times(Asc, 32 + r, 0, Tsc, 0, c4, 32));
  }
  __syncthreads();
  {
    const int r = tid >> 3, c4 = (tid & 7) * 4;
    const float4 y = row_times(Tsc, 32 + r, 32, Asc, 0, 32 + c4, 32);
    put_row4(Tsc, 32 + r, c4, make_float4(-y.x, -y.y, -y.z, -y.w));
  }
  __syncthreads();
}

template <bool kLo>
__global__ void __launch_bounds__(kThreads, 1)
    gdn_chunk_kernel(float *__restrict__ S, const float *__restrict__ q,
                     const float *__restrict__ k, const float *__restrict__ v,
                     const float *__restrict__ g,
                     const float *__restrict__ beta, float *__restrict__ o,
                     int T, int kh, int vh, int rep) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw_s = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t sb = (raw_s + 1023u) & ~1023u;
  unsigned char *gb = smem_raw + (sb - raw_s);
  float *Gam = reinterpret_cast<float *>(gb + OFF_VEC);
  float *gam = Gam + 64;
  float *wv = Gam + 128;
  float *bet = Gam + 192;
  float *gam_o = Gam + 256;       // [2][64]: gamma of the chunk whose o is pending
  const uint32_t bar0 = sb + OFF_BAR;
  volatile uint32_t *slot = reinterpret_cast<volatile uint32_t *>(gb + OFF_BAR + 32);
  float *Asc = reinterpret_cast<float *>(gb + OFF_SCR);
  float *Tsc = Asc + 64 * 64;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3;      // TMEM lane quadrant of this warp
  const int half = warp >> 2;     // which half of the columns this warp moves
  const int myrow = 32 * quad + lane;
  const uint32_t lane_base = (uint32_t)(32 * quad) << 16;

  const int head = blockIdx.x;
  const int b = head / vh, vi = head % vh, hh = vi / rep;
  const size_t head_off = (size_t)head * kD * kD;
  const int nchunks = (T + kC - 1) / kC;

  const Operand opKQ{sb + OFF_KQ, 128, 128, false};   // MMA-a A
  const Operand opKb{sb + OFF_KQ, 128, 128, false};   // MMA-a B (rows 0-63)
  const Operand opKmn{sb + OFF_KQ, 128, 128, true};   // MMA-w A (rows 0-63)
  const Operand opVmn{sb + OFF_V, 64, 128, true};     // MMA-u A
  const Operand opTB{sb + OFF_TB, 64, 64, false};     // MMA-w B
  const Operand opTB2{sb + OFF_TB2, 64, 64, false};   // MMA-u B
  const Operand opST{sb + OFF_ST, 128, 128, false};   // MMA-1 A
  const Operand opWT{sb + OFF_WT, 128, 64, true};     // MMA-1 B (W part)
  const Operand opQb{sb + OFF_KQ + 64 * 128, 128, 128, false};  // MMA-1 B (Q rows)
  const Operand opDT{sb + OFF_DT, 128, 64, false};    // MMA-3 A
  const Operand opP{sb + OFF_P, 64, 64, false};       // MMA-3 B
  const Operand opDTW{sb + OFF_DTW, 128, 64, false};  // MMA-4 A
  const Operand opKnB{sb + OFF_KQ, 128, 128, true};   // MMA-4 B (K rows)

  if (warp == 0) tmem_alloc(sb + OFF_BAR + 32, 512);
  if (tid == 0)
    for (int i = 0; i < 4; ++i) mbar_init(bar0 + 8 * i, 1);
  cta_sync_tc();
  const uint32_t tmem = *slot;
  const uint32_t tl = tmem + lane_base;

  // Inputs of one chunk held in registers: rows (tid >> 4) + 16 i of
  // [K; Q; V] (i = 0..11), columns (tid & 15) * 8 .. + 7; and, on warp 0,
  // the gates of tokens lane and lane + 32.
  float4 pre[24];
  float pg[2], pb[2];
  auto prefetch = [&](int c) {
    const int t0 = c * kC;
    const int n = min(kC, T - t0);
    const size_t qk_base = ((size_t)b * T + t0) * kh + hh;
    const size_t v_base = ((size_t)b * T + t0) * vh + vi;
    const int c0 = (tid & 15) * 8;
#pragma unroll
    for (int i = 0; i < 12; ++i) {
      const int row = (tid >> 4) + 16 * i;
      const int t = row & (kC - 1);
      const float *src = i < 4 ? k : (i < 8 ? q : v);
      if (t < n) {
        const size_t base = i < 8 ? (qk_base + (size_t)t * kh) * kD
                                  : (v_base + (size_t)t * vh) * kD;
        pre[2 * i] = __ldg(reinterpret_cast<const float4 *>(src + base + c0));
        pre[2 * i + 1] = __ldg(reinterpret_cast<const float4 *>(src + base + c0 + 4));
      } else {
        pre[2 * i] = make_float4(0.f, 0.f, 0.f, 0.f);
        pre[2 * i + 1] = pre[2 * i];
      }
    }
    if (warp == 0) {
      pg[0] = lane < n ? __ldg(g + v_base + (size_t)lane * vh) : 0.f;
      pg[1] = lane + 32 < n ? __ldg(g + v_base + (size_t)(lane + 32) * vh) : 0.f;
      pb[0] = lane < n ? __ldg(beta + v_base + (size_t)lane * vh) : 0.f;
      pb[1] = lane + 32 < n ? __ldg(beta + v_base + (size_t)(lane + 32) * vh) : 0.f;
    }
  };
  prefetch(0);

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
  cta_sync_tc();

  // o for chunk cc = diag(gamma) (Q S)^T + (P Delta)^T, read from TMEM.
  auto emit_o = [&](int cc) {
    const int nn = min(kC, T - cc * kC);
    const size_t vb = ((size_t)b * T + (size_t)cc * kC) * vh + vi;
    const float *gm = gam_o + (cc & 1) * 64;
    for (int c0 = half * 32; c0 < half * 32 + 32; c0 += 16) {
      float r[16], pd[16];
      tmem_ld16(tl + T_QS + c0, r);
      tmem_ld16(tl + T_PD + c0, pd);
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const int t = c0 + jj;
        if (t < nn) o[(vb + (size_t)t * vh) * kD + myrow] = fmaf(gm[t], r[jj], pd[jj]);
      }
    }
  };

  uint32_t parity = 0;
  bool failed = false;
  for (int c = 0; c < nchunks; ++c) {
    // ------------------------------------------ phase 0: inputs, S^T operand
    if (warp == 0) {
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
      gam_o[(c & 1) * 64 + lane] = gam[lane];
      gam_o[(c & 1) * 64 + lane + 32] = gam[lane + 32];
      wv[lane] = expf(last - sa);
      wv[lane + 32] = expf(last - sc);
    }
    // [K; Q] rows and V rows from the prefetched registers.
#pragma unroll
    for (int i = 0; i < 12; ++i) {
      const int row = (tid >> 4) + 16 * i, c0 = (tid & 15) * 8;
      const float x[8] = {pre[2 * i].x, pre[2 * i].y, pre[2 * i].z, pre[2 * i].w,
                          pre[2 * i + 1].x, pre[2 * i + 1].y, pre[2 * i + 1].z,
                          pre[2 * i + 1].w};
      if (i < 8)
        put8<kLo>(gb, OFF_KQ, 128, 128, row, c0, x);
      else
        put8<kLo>(gb, OFF_V, 64, 128, row & (kC - 1), c0, x);
    }
    // S^T operand (rows dv, columns dk) from the TMEM master copy.
    for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 16) {
      float r[16];
      tmem_ld16(tl + T_SACC + c0, r);
      put8<kLo>(gb, OFF_ST, 128, 128, myrow, c0, r);
      put8<kLo>(gb, OFF_ST, 128, 128, myrow, c0 + 8, r + 8);
    }
    fence_proxy_async();
    cta_sync_tc();

    // --------------------------------------- phase 1: G, H = [K;Q] K^T
    if (tid == 0) {
      gemm<kLo>(tmem + T_GH, opKQ, opKb, 128, kC, kD / 16, false);
      commit(bar0);
    }
    if (c > 0) emit_o(c - 1);  // the previous chunk's output, under this product
    if (!__syncthreads_and(mbar_wait(bar0, parity, kWaitLimit))) { failed = true; break; }
    fence_after_sync();

    // -------------------------- phase 2: A, T = (I + A)^-1, T diag operands
    if (quad < 2) {  // lanes 0-63 hold G rows t
      const int t = myrow;
      const float bt = bet[t], Gt = Gam[t];
      for (int c0 = half * 32; c0 < half * 32 + 32; c0 += 16) {
        float r[16];
        tmem_ld16(tl + T_GH + c0, r);
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
          float4 a4;
          float *a = &a4.x;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int s = c0 + 4 * j4 + e;
            a[e] = s < t ? bt * expf(Gt - Gam[s]) * r[4 * j4 + e] : 0.f;
          }
          *reinterpret_cast<float4 *>(Asc + sidx(t, c0 + 4 * j4)) = a4;
        }
      }
    }
    if (quad >= 2) {  // lanes 64-127 hold H rows t: P in place of H
      const int t = myrow - kC;
      const float Gt = Gam[t];
      for (int c0 = half * 32; c0 < half * 32 + 32; c0 += 16) {
        float r[16];
        tmem_ld16(tl + T_GH + c0, r);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int s = c0 + e;
          r[e] = s <= t ? expf(Gt - Gam[s]) * r[e] : 0.f;
        }
        tmem_st16(tl + T_GH + c0, r);
      }
    }
    __syncthreads();
    tri_inverse(Asc, Tsc, tid);
    {
      // each thread takes one row-half of T: row t = tid >> 2, 16 columns
      const int t = tid >> 2, cq = (tid & 3) * 16;
      float tr[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) tr[e] = Tsc[sidx(t, cq + e)];
      __syncthreads();  // everyone holds its T values; scratch may be reused
      float x1[8], x2[8];
#pragma unroll
      for (int h8 = 0; h8 < 2; ++h8) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int s = cq + 8 * h8 + e;
          x1[e] = tr[8 * h8 + e] * bet[s] * gam[s];
          x2[e] = tr[8 * h8 + e] * bet[s];
        }
        put8<kLo>(gb, OFF_TB, kC, kC, t, cq + 8 * h8, x1);
        put8<kLo>(gb, OFF_TB2, kC, kC, t, cq + 8 * h8, x2);
      }
    }
    fence_proxy_async();
    cta_sync_tc();

    // ------------------------------------------------ phase 3: W^T, U^T
    if (tid == 0) {
      gemm<kLo>(tmem + T_W, opKmn, opTB, 128, kC, kC / 16, false);
      gemm<kLo>(tmem + T_U, opVmn, opTB2, 128, kC, kC / 16, false);
      commit(bar0 + 8);
    }
    if (!__syncthreads_and(mbar_wait(bar0 + 8, parity, kWaitLimit))) { failed = true; break; }
    fence_after_sync();

    // ------------------------------------------- phase 4: W^T operand
    for (int c0 = half * 32; c0 < half * 32 + 32; c0 += 16) {
      float r[16];
      tmem_ld16(tl + T_W + c0, r);  // lane dk, columns t
      put8<kLo>(gb, OFF_WT, 128, kC, myrow, c0, r);
      put8<kLo>(gb, OFF_WT, 128, kC, myrow, c0 + 8, r + 8);
    }
    fence_proxy_async();
    cta_sync_tc();

    // ----------------------------- phase 5: (W S)^T, (Q S)^T = S^T [W^T | Q^T]
    if (tid == 0) {
      gemm<kLo>(tmem + T_U, opST, opWT, 128, kC, kD / 16, true, true);
      gemm<kLo>(tmem + T_QS, opST, opQb, 128, kC, kD / 16, false);
      commit(bar0 + 16);
    }
    if (!__syncthreads_and(mbar_wait(bar0 + 16, parity, kWaitLimit))) { failed = true; break; }
    fence_after_sync();

    // ---- phase 6: Delta^T = U^T - (W S)^T, Delta^T diag(w); P; S^T *= gamma_63
    for (int c0 = half * 32; c0 < half * 32 + 32; c0 += 16) {
      float u[16];
      tmem_ld16(tl + T_U + c0, u);  // Delta^T = U^T - (W S)^T
      put8<kLo>(gb, OFF_DT, 128, kC, myrow, c0, u);
      put8<kLo>(gb, OFF_DT, 128, kC, myrow, c0 + 8, u + 8);
#pragma unroll
      for (int e = 0; e < 16; ++e) u[e] *= wv[c0 + e];
      put8<kLo>(gb, OFF_DTW, 128, kC, myrow, c0, u);
      put8<kLo>(gb, OFF_DTW, 128, kC, myrow, c0 + 8, u + 8);
    }
    if (quad >= 2) {  // lanes 64-127 hold P rows t (built in phase 2)
      const int t = myrow - kC;
      for (int c0 = half * 32; c0 < half * 32 + 32; c0 += 16) {
        float r[16];
        tmem_ld16(tl + T_GH + c0, r);
        put8<kLo>(gb, OFF_P, kC, kC, t, c0, r);
        put8<kLo>(gb, OFF_P, kC, kC, t, c0 + 8, r + 8);
      }
    }
    {
      const float gC = gam[kC - 1];
      for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 16) {
        float r[16];
        tmem_ld16(tl + T_SACC + c0, r);
#pragma unroll
        for (int j = 0; j < 16; ++j) r[j] *= gC;
        tmem_st16(tl + T_SACC + c0, r);
      }
    }
    fence_proxy_async();
    cta_sync_tc();

    // ---------- phase 7: (P Delta)^T = Delta^T P^T; S^T += Delta^T diag(w) K
    if (tid == 0) {
      gemm<kLo>(tmem + T_PD, opDT, opP, 128, kC, kC / 16, false);
      gemm<kLo>(tmem + T_SACC, opDTW, opKnB, 128, kD, kC / 16, true);
      commit(bar0 + 24);
    }
    if (c + 1 < nchunks) prefetch(c + 1);  // overlaps the products above
    if (!__syncthreads_and(mbar_wait(bar0 + 24, parity, kWaitLimit))) { failed = true; break; }
    fence_after_sync();

    cta_sync_tc();
    parity ^= 1u;
  }

  if (!failed) {
    emit_o(nchunks - 1);
    float *Sh = S + head_off;
    for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 16) {
      float r[16];
      tmem_ld16(tl + T_SACC + c0, r);
#pragma unroll
      for (int j = 0; j < 16; ++j) Sh[(size_t)(c0 + j) * kD + myrow] = r[j];
    }
  } else if (tid == 0) {
    atomicAdd(&g_prefill_timeouts, 1u);
  }
  cta_sync_tc();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

size_t prefill_workspace_bytes(int, int, int, int, int, int) { return 0; }

cudaError_t launch_prefill_chunked(float *S, const float *q, const float *k,
                                   const float *v, const float *g,
                                   const float *beta, float *o, int B, int kh,
                                   int vh, int T, int precision, void *,
                                   cudaStream_t stream) {
  const size_t nheads = (size_t)B * vh;
  if (nheads == 0) return cudaSuccess;
  if (nheads > 0x7fffffffull) return cudaErrorInvalidConfiguration;
  cudaError_t e;
  if (precision == 1) {
    e = cudaFuncSetAttribute(gdn_chunk_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    gdn_chunk_kernel<true><<<(unsigned)nheads, kThreads, kSmemAlloc, stream>>>(
        S, q, k, v, g, beta, o, T, kh, vh, vh / kh);
  } else {
    e = cudaFuncSetAttribute(gdn_chunk_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    gdn_chunk_kernel<false><<<(unsigned)nheads, kThreads, kSmemAlloc, stream>>>(
        S, q, k, v, g, beta, o, T, kh, vh, vh / kh);
  }
  return cudaGetLastError();
}

cudaError_t prefill_timeouts(unsigned int *count) {
  return cudaMemcpyFromSymbol(count, g_prefill_timeouts, sizeof(unsigned int));
}

}  // namespace gdn
