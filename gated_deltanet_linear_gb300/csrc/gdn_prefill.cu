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
// Everything is computed in the transposed orientation so that the value /
// key dimension (128) is the MMA's M and the state lives in tensor memory as
// S^T with one TMEM lane per value column.
//
// One CTA per (sequence, value head) walks the chunks in order; the fp32
// master copy of S^T stays in TMEM for the whole sequence.  Per chunk:
//   MMA-a  [K;Q] K^T           -> G = K K^T, H = Q K^T           (TMEM)
//   SIMT   A from G, T = (I+A)^-1 by column-parallel forward substitution
//   MMA-d  K^T (T diag(beta gamma))^T -> W^T,  V^T (T diag(beta))^T -> U^T
//   MMA-1  S^T [W; diag(gamma) Q]^T -> (W S)^T, (diag(gamma) Q S)^T
//   SIMT   Delta^T = U^T - (W S)^T;  S^T *= gamma_63 in TMEM
//   MMA-3  (diag(gamma) Q S)^T += Delta^T P^T     -> O^T
//   MMA-4  S^T += Delta^T (diag(w) K)               -> next chunk's S^T
//
// Precision.  Operands live in shared memory in one of two formats:
//   split-bf16 ("BF16X3"): x = hi + lo with hi = bf16(x), lo = bf16(x - hi);
//     a product is hi*hi + hi*lo + lo*hi, three bf16 MMAs with fp32
//     accumulation (about 16 significant bits per operand, relative error
//     ~1e-5 on the results);
//   TF32: x rounded to tf32 (10 explicit mantissa bits), one tf32 MMA
//     (relative error ~1e-3).
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

// Shared memory (byte offsets from a 1024-aligned base).  Operand tiles
// hold R x K elements in 4 bytes each (fp32, or bf16 hi tile + bf16 lo tile).
constexpr uint32_t OFF_KQ = 0;         // 128 x 128: [K; Q], later [W; gamma Q]
constexpr uint32_t OFF_KT = 65536;     // 128 x 64: K^T, later (diag(w) K)^T
constexpr uint32_t OFF_VT = 98304;     // 128 x 64: V^T, later Delta^T
constexpr uint32_t OFF_TB = 131072;    // 64 x 64: T diag(beta gamma) (and A scratch)
constexpr uint32_t OFF_TB2 = 147456;   // 64 x 64: T diag(beta), later P
constexpr uint32_t OFF_ST = 163840;    // 128 x 128: S^T
constexpr uint32_t OFF_VEC = 229376;   // Gamma, gamma, w, beta: 4 x 64 floats
constexpr uint32_t OFF_BAR = 230400;   // 4 mbarriers, TMEM address
constexpr uint32_t kSmemUsed = OFF_BAR + 64;
constexpr uint32_t kSmemAlloc = kSmemUsed + 1024;  // room to align the base

// TMEM columns (512 allocated).
constexpr uint32_t T_SACC = 0;    // S^T, fp32 master (128 columns = dk)
constexpr uint32_t T_GH = 128;    // G (lanes 0-63), H (lanes 64-127): 64 columns
constexpr uint32_t T_W = 192;     // W^T: lanes dk, columns t
constexpr uint32_t T_U = 256;     // U^T: lanes dv, columns t
constexpr uint32_t T_D1 = 320;    // (W S)^T: lanes dv, columns t
constexpr uint32_t T_O = 384;     // (gamma Q S)^T + Delta^T P^T = O^T

constexpr uint32_t kWaitLimit = 1u << 24;

__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 v) {
  return *reinterpret_cast<uint32_t *>(&v);
}

// Store 4 consecutive K elements (k0 % 4 == 0) of row r of an R x K tile.
template <bool kBF16>
__device__ __forceinline__ void put4(unsigned char *gb, uint32_t off, int R,
                                     int K, int r, int k0, float4 x) {
  if (kBF16) {
    const __nv_bfloat162 h01 = __floats2bfloat162_rn(x.x, x.y);
    const __nv_bfloat162 h23 = __floats2bfloat162_rn(x.z, x.w);
    const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
    const __nv_bfloat162 l01 = __floats2bfloat162_rn(x.x - f01.x, x.y - f01.y);
    const __nv_bfloat162 l23 = __floats2bfloat162_rn(x.z - f23.x, x.w - f23.y);
    const uint32_t o = off + sw128_off(R, r, k0, 2);
    *reinterpret_cast<uint2 *>(gb + o) = make_uint2(bf2_bits(h01), bf2_bits(h23));
    *reinterpret_cast<uint2 *>(gb + o + (uint32_t)(R * K * 2)) =
        make_uint2(bf2_bits(l01), bf2_bits(l23));
  } else {
    *reinterpret_cast<float4 *>(gb + off + sw128_off(R, r, k0, 4)) =
        make_float4(to_tf32(x.x), to_tf32(x.y), to_tf32(x.z), to_tf32(x.w));
  }
}

template <bool kBF16>
__device__ __forceinline__ void put1(unsigned char *gb, uint32_t off, int R,
                                     int K, int r, int k, float x) {
  if (kBF16) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
    const uint32_t o = off + sw128_off(R, r, k, 2);
    *reinterpret_cast<__nv_bfloat16 *>(gb + o) = h;
    *reinterpret_cast<__nv_bfloat16 *>(gb + o + (uint32_t)(R * K * 2)) = l;
  } else {
    *reinterpret_cast<float *>(gb + off + sw128_off(R, r, k, 4)) = to_tf32(x);
  }
}

// D[M][N] (+)= A[M][K] B[N][K]^T with A an aR x K tile at a, B a bR x K tile
// at b (the first N rows are used).  Issued by one thread.
template <bool kBF16>
__device__ __forceinline__ void gemm(uint32_t d, uint32_t a, int aR,
                                     uint32_t b, int bR, int K, int M, int N,
                                     bool accumulate) {
  if (kBF16) {
    const uint32_t id = idesc(kFmtBF16, M, N);
    const uint32_t a_lo = a + (uint32_t)(aR * K * 2);
    const uint32_t b_lo = b + (uint32_t)(bR * K * 2);
    for (int ks = 0; ks < K / 16; ++ks) {
      const uint64_t ah = desc_kstep(a, aR, ks), bh = desc_kstep(b, bR, ks);
      mma_bf16(d, ah, bh, id, (accumulate || ks > 0) ? 1u : 0u);
      mma_bf16(d, ah, desc_kstep(b_lo, bR, ks), id, 1u);
      mma_bf16(d, desc_kstep(a_lo, aR, ks), bh, id, 1u);
    }
  } else {
    const uint32_t id = idesc(kFmtTF32, M, N);
    for (int ks = 0; ks < K / 8; ++ks)
      mma_tf32(d, desc_kstep(a, aR, ks), desc_kstep(b, bR, ks), id,
               (accumulate || ks > 0) ? 1u : 0u);
  }
}

__device__ __forceinline__ void cta_sync_tc() {
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
}

template <bool kBF16>
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
  const uint32_t bar0 = sb + OFF_BAR;
  volatile uint32_t *slot = reinterpret_cast<volatile uint32_t *>(gb + OFF_BAR + 32);

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

  if (warp == 0) tmem_alloc(sb + OFF_BAR + 32, 512);
  if (tid == 0)
    for (int i = 0; i < 4; ++i) mbar_init(bar0 + 8 * i, 1);
  cta_sync_tc();
  const uint32_t tmem = *slot;

  // State in: S[dk][dv] -> TMEM lane dv, column dk.
  {
    const float *Sh = S + head_off;
    for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 16) {
      float r[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) r[j] = __ldg(Sh + (size_t)(c0 + j) * kD + myrow);
      tmem_st16(tmem + lane_base + T_SACC + c0, r);
    }
  }
  cta_sync_tc();

  uint32_t parity = 0;
  bool failed = false;
  for (int c = 0; c < nchunks; ++c) {
    const int t0 = c * kC;
    const int n = min(kC, T - t0);
    const size_t qk_base = ((size_t)b * T + t0) * kh + hh;   // row of token t0
    const size_t v_base = ((size_t)b * T + t0) * vh + vi;

    // ---------------------------------------------------------- phase 0
    if (warp == 0) {
      const float ga = lane < n ? __ldg(g + v_base + (size_t)lane * vh) : 0.f;
      const float gb2 = lane + 32 < n ? __ldg(g + v_base + (size_t)(lane + 32) * vh) : 0.f;
      bet[lane] = lane < n ? __ldg(beta + v_base + (size_t)lane * vh) : 0.f;
      bet[lane + 32] = lane + 32 < n ? __ldg(beta + v_base + (size_t)(lane + 32) * vh) : 0.f;
      float sa = ga, sc = gb2;
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
    }
    // [K; Q] rows (token-major), one row per warp iteration, 4 elements/lane.
    for (int rr = warp; rr < 2 * kC; rr += kThreads / 32) {
      const int t = rr & (kC - 1);
      const float *src = rr < kC ? k : q;
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < n)
        x = __ldg(reinterpret_cast<const float4 *>(
            src + (qk_base + (size_t)t * kh) * kD + 4 * lane));
      put4<kBF16>(gb, OFF_KQ, 128, 128, rr, 4 * lane, x);
    }
    // K^T and V^T: thread owns row r (dk or dv), 4 tokens per store.
    {
      const int r = tid & 127;
      for (int t4 = (tid >> 7) * 4; t4 < kC; t4 += 8) {
        float kx[4], vx[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int t = t4 + j;
          kx[j] = t < n ? __ldg(k + (qk_base + (size_t)t * kh) * kD + r) : 0.f;
          vx[j] = t < n ? __ldg(v + (v_base + (size_t)t * vh) * kD + r) : 0.f;
        }
        put4<kBF16>(gb, OFF_KT, 128, kC, r, t4, make_float4(kx[0], kx[1], kx[2], kx[3]));
        put4<kBF16>(gb, OFF_VT, 128, kC, r, t4, make_float4(vx[0], vx[1], vx[2], vx[3]));
      }
    }
    // S^T operand from the TMEM master copy.
    for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 16) {
      float r[16];
      tmem_ld16(tmem + lane_base + T_SACC + c0, r);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        put4<kBF16>(gb, OFF_ST, 128, 128, myrow, c0 + 4 * i,
                    make_float4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]));
    }
    fence_proxy_async();
    cta_sync_tc();

    // ------------------------------------------- phase 1: G, H = [K;Q] K^T
    if (tid == 0) {
      gemm<kBF16>(tmem + T_GH, sb + OFF_KQ, 128, sb + OFF_KQ, 128, kD, 128, kC, false);
      commit(bar0);
    }
    if (!__syncthreads_and(mbar_wait(bar0, parity, kWaitLimit))) { failed = true; break; }
    fence_after_sync();

    // ------------------------------- phase 2: A and T = (I + A)^-1 (fp32)
    // A scratch, fp32 [64][64], permuted so that the 16 entries a solver
    // thread needs for one row are contiguous: (t, s) -> t*64 + (s&3)*16 + s/4.
    float *Asc = reinterpret_cast<float *>(gb + OFF_TB);
    if (quad < 2) {
      const int t = myrow;
      for (int c0 = half * 32; c0 < half * 32 + 32; c0 += 16) {
        float r[16];
        tmem_ld16(tmem + lane_base + T_GH + c0, r);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int s = c0 + j;
          const float a = s < t ? bet[t] * expf(Gam[t] - Gam[s]) * r[j] : 0.f;
          Asc[t * 64 + (s & 3) * 16 + (s >> 2)] = a;
        }
      }
    }
    __syncthreads();
    float x[16];
    {
      // Column j of T, rows split over 4 lanes by t mod 4.
      const int j = tid >> 2, q4 = tid & 3;
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = 0.f;
#pragma unroll
      for (int t = 0; t < kC; ++t) {
        const float4 *arow = reinterpret_cast<const float4 *>(Asc + t * 64 + q4 * 16);
        float part = 0.f;
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) {
          const float4 a = arow[i4];
          part = fmaf(a.x, x[4 * i4 + 0], part);
          part = fmaf(a.y, x[4 * i4 + 1], part);
          part = fmaf(a.z, x[4 * i4 + 2], part);
          part = fmaf(a.w, x[4 * i4 + 3], part);
        }
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        const float xt = (t == j ? 1.f : 0.f) - part;
        if ((t & 3) == q4) x[t >> 2] = xt;
      }
    }
    __syncthreads();  // everyone is done with the A scratch
    {
      const int j = tid >> 2, q4 = tid & 3;
      const float bg = bet[j] * gam[j], bj = bet[j];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int t = q4 + 4 * i;
        put1<kBF16>(gb, OFF_TB, kC, kC, t, j, x[i] * bg);
        put1<kBF16>(gb, OFF_TB2, kC, kC, t, j, x[i] * bj);
      }
    }
    fence_proxy_async();
    cta_sync_tc();

    // ------------------------------------------------- phase 3: W^T, U^T
    if (tid == 0) {
      gemm<kBF16>(tmem + T_W, sb + OFF_KT, 128, sb + OFF_TB, kC, kC, 128, kC, false);
      gemm<kBF16>(tmem + T_U, sb + OFF_VT, 128, sb + OFF_TB2, kC, kC, 128, kC, false);
      commit(bar0 + 8);
    }
    if (!__syncthreads_and(mbar_wait(bar0 + 8, parity, kWaitLimit))) { failed = true; break; }
    fence_after_sync();

    // ----------------- phase 4: [W; gamma Q], (diag(w) K)^T and P operands
    for (int c0 = half * 32; c0 < half * 32 + 32; c0 += 16) {
      float r[16];
      tmem_ld16(tmem + lane_base + T_W + c0, r);  // lane dk, columns t
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) put1<kBF16>(gb, OFF_KQ, 128, 128, c0 + jj, myrow, r[jj]);
    }
    for (int t = warp; t < kC; t += kThreads / 32) {
      float4 x4 = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < n) {
        x4 = __ldg(reinterpret_cast<const float4 *>(
            q + (qk_base + (size_t)t * kh) * kD + 4 * lane));
        const float gt = gam[t];
        x4.x *= gt; x4.y *= gt; x4.z *= gt; x4.w *= gt;
      }
      put4<kBF16>(gb, OFF_KQ, 128, 128, kC + t, 4 * lane, x4);
    }
    {
      const int r = tid & 127;
      for (int t4 = (tid >> 7) * 4; t4 < kC; t4 += 8) {
        float kx[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int t = t4 + j;
          kx[j] = t < n ? __ldg(k + (qk_base + (size_t)t * kh) * kD + r) * wv[t] : 0.f;
        }
        put4<kBF16>(gb, OFF_KT, 128, kC, r, t4, make_float4(kx[0], kx[1], kx[2], kx[3]));
      }
    }
    if (quad >= 2) {
      const int t = myrow - kC;
      for (int c0 = half * 32; c0 < half * 32 + 32; c0 += 16) {
        float r[16];
        tmem_ld16(tmem + lane_base + T_GH + c0, r);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float pv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int s = c0 + 4 * i + e;
            pv[e] = s <= t ? expf(Gam[t] - Gam[s]) * r[4 * i + e] : 0.f;
          }
          put4<kBF16>(gb, OFF_TB2, kC, kC, t, c0 + 4 * i, make_float4(pv[0], pv[1], pv[2], pv[3]));
        }
      }
    }
    fence_proxy_async();
    cta_sync_tc();

    // ---------------------------- phase 5: S^T [W; gamma Q]^T -> D1, O
    if (tid == 0) {
      gemm<kBF16>(tmem + T_D1, sb + OFF_ST, 128, sb + OFF_KQ, 128, kD, 128, 2 * kC, false);
      commit(bar0 + 16);
    }
    if (!__syncthreads_and(mbar_wait(bar0 + 16, parity, kWaitLimit))) { failed = true; break; }
    fence_after_sync();

    // ------------------- phase 6: Delta^T = U^T - (W S)^T; S^T *= gamma_63
    for (int c0 = half * 32; c0 < half * 32 + 32; c0 += 16) {
      float u[16], d[16];
      tmem_ld16(tmem + lane_base + T_U + c0, u);
      tmem_ld16(tmem + lane_base + T_D1 + c0, d);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        put4<kBF16>(gb, OFF_VT, 128, kC, myrow, c0 + 4 * i,
                    make_float4(u[4 * i] - d[4 * i], u[4 * i + 1] - d[4 * i + 1],
                                u[4 * i + 2] - d[4 * i + 2], u[4 * i + 3] - d[4 * i + 3]));
    }
    {
      const float gC = gam[kC - 1];
      for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 16) {
        float r[16];
        tmem_ld16(tmem + lane_base + T_SACC + c0, r);
#pragma unroll
        for (int j = 0; j < 16; ++j) r[j] *= gC;
        tmem_st16(tmem + lane_base + T_SACC + c0, r);
      }
    }
    fence_proxy_async();
    cta_sync_tc();

    // -------------------- phase 7: O^T += Delta^T P^T; S^T += Delta^T K~
    if (tid == 0) {
      gemm<kBF16>(tmem + T_O, sb + OFF_VT, 128, sb + OFF_TB2, kC, kC, 128, kC, true);
      gemm<kBF16>(tmem + T_SACC, sb + OFF_VT, 128, sb + OFF_KT, 128, kC, 128, kD, true);
      commit(bar0 + 24);
    }
    if (!__syncthreads_and(mbar_wait(bar0 + 24, parity, kWaitLimit))) { failed = true; break; }
    fence_after_sync();

    // ------------------------------------------------ phase 8: o out
    for (int c0 = half * 32; c0 < half * 32 + 32; c0 += 16) {
      float r[16];
      tmem_ld16(tmem + lane_base + T_O + c0, r);
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const int t = c0 + jj;
        if (t < n) o[(v_base + (size_t)t * vh) * kD + myrow] = r[jj];
      }
    }
    cta_sync_tc();
    parity ^= 1u;
  }

  if (!failed) {
    float *Sh = S + head_off;
    for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 16) {
      float r[16];
      tmem_ld16(tmem + lane_base + T_SACC + c0, r);
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
