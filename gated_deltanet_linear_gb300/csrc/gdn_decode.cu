// Token-serial gated delta-rule update for sm_103a (decode, M-token verify,
// fp32 prefill).
//
// What it computes (per sequence b, value head vi, key head hh = vi / rep,
// token m), "Kestrel_VLLM - 24 · GDN linear attention to GPU", section 4:
//     alpha = exp(g);  S = alpha S;  kv = S^T k;  tmp = (v - kv) beta;
//     S = S + k tmp^T;  o = S^T q.
// The output is taken in the algebraically equal form
//     o = alpha (S_old^T q) + (q . k) tmp,
// so that S^T k, S^T q and q . k come out of one pass over the state and
// the rank-1 update follows; the state after the update is the same
// expression as in the definition.
//
// Work split.  A head's 128 x 128 state is 64 KB.  A work unit is one head's
// value columns [8c, 8c+8) over all 128 key rows (4 KB), so every reduction
// over the key dimension stays inside one warp (no barriers):
//   lane = 2 * p + h,  p in 0..15 -> key rows 8p .. 8p+7,
//                      h in 0..1  -> value columns 8c + 4h .. 8c + 4h + 3.
// Each lane keeps its 8 x 4 block of S in registers for all M tokens, so
// the state is read from HBM once and written once per launch however many
// tokens it covers (the register-resident idea of "27 · register-resident &
// fused launch", section 3, split over 16 warps instead of one thread per
// column).
//
// Memory pipeline.  The kernel is persistent (16 warps per SM, bound by
// registers and shared memory, in CTAs of 4 warps, or of 8 for one token
// read from host memory): each warp walks a strided list
// of units and keeps the next kStages - 1 of them in flight with cp.async
// (16 bytes per lane per row, L2-only) into a private ring of 4 KB stages in
// shared memory, so HBM reads continue while the warp computes.  A lane reads
// back only the bytes it copied itself, so no barrier is needed; the stage
// layout is XOR-swizzled so the 128-bit shared loads of a quarter warp hit
// eight distinct 16-byte bank groups.  One warp instruction touches 16 full
// 32-byte sectors of global memory.  Results go straight from registers to
// global memory with 128-bit stores that skip L1 (for one token, also
// leaving the line's L2 eviction priority unchanged).
//
// Launch overlap.  Behind the layer prologue the kernel is launched as a
// programmatic dependent: it may start while the prologue still runs, puts
// its first state units in flight (the prologue never writes the state),
// and waits for the prologue's results (griddepcontrol.wait) before its
// first read of the token inputs.  A single-token launch that fills every
// CTA slot is a programmatic dependent of whatever kernel came before (the
// previous decode step, which writes the state): its CTAs are launched as
// the previous kernel's CTAs leave, and wait for that kernel's end before
// they read anything.  In an ordinary launch the wait returns at once.  The
// kernels let their own dependents be scheduled once every CTA (or warp)
// has reached its last unit; those wait for the completion in the same way
// before reading the outputs.  Signalled at the start instead, a following
// layer prologue's small CTAs waited beside the running update for its
// whole length and slowed it (64 x 48-head layer step: 90.0 us against
// 67.9 us).
//
// Three layouts share that arithmetic:
//   - gdn_step_c32_kernel: single-token launches (with host-memory
//     inputs, CTAs of two column groups of a head).  A CTA of 4 warps takes a 32-column group of a head, warp w
//     key rows 32w .. 32w+31 of all 32 columns, so every warp request covers
//     whole 128-byte row segments; the reductions over the key rows finish
//     across the 4 warps through shared memory, one barrier per unit.  On
//     the 64 x 48-head step it measured 65.1 us against 69.7 us for the
//     8-column layout.
//   - gdn_steps_head_kernel: several tokens without checkpoints, with
//     device-resident inputs.  One CTA of 8 warps per head, 16 columns per
//     warp, two 8-row blocks per lane; the token inputs stream through a
//     shared-memory ring filled by bulk copies (see its comment).  On
//     64 x 48 heads it measured 73 / 79 / 121 us for M = 2 / 4 / 8,
//     against 82 / 109 / 170 us for the 8-column layout.
//   - gdn_steps_kernel (the 8-column layout above): checkpointing launches
//     (bound by their stores, faster here), multi-token launches whose
//     token inputs are in host memory (8 warps on neighbouring column groups
//     share a head's q and k rows in L1), and those of fewer heads than SMs.
//
// Determinism.  Every product and sum is an explicit round-to-nearest
// intrinsic and the reduction tree is fixed, so a token gives the same bits
// whether it is the only token of a launch or one of M, and in any of the
// layouts: gdn_step_m(M) is bit-identical to M gdn_step calls.  The tree over
// the 16 blocks of 8 key rows (block p = rows 8p .. 8p+7, each summed in row
// order): W_w = (B_4w + B_4w+2) + (B_4w+1 + B_4w+3) for w = 0..3, then
// (W_0 + W_2) + (W_1 + W_3); q . k the same way.

#include "gdn_internal.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int kStages = 3;        // cp.async ring depth per warp
constexpr int kWarpsPerSm = 16;   // bound by registers and shared memory
constexpr int kUnitsPerHead = kDim / 8;          // 16 column groups
constexpr int kUnitFloats = kDim * 8;            // 4 KB
// Warps per CTA: 4, or 8 for checkpointing single-token launches whose token
// inputs are in host memory, so that the 8 warps working on neighbouring
// column groups of a head share its q and k rows in one SM's L1 (a 64 x
// 48-head step took 70 us instead of 86 us that way; with device inputs
// 4-warp CTAs are 0.2 % faster, and 8 measured 2-7 % slower for several
// tokens).
template <int kWarps>
__host__ __device__ constexpr int smem_per_cta() {
  return kWarps * kStages * kUnitFloats * 4;
}
constexpr unsigned kFull = 0xffffffffu;

// L2 policy for the single-token state stores: the written line keeps the
// eviction priority it had (in place, the line the same warp has just
// read).  On the batched decode step in place this measured 70.3 -> 69.5 us
// against a plain store; the multi-token launches, at their register limit,
// were 2-4 % slower with it and keep the plain store.
__device__ __forceinline__ uint64_t l2_keep_priority() {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_unchanged.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

template <bool kHint>
__device__ __forceinline__ void st_stream(float *p, float4 v, uint64_t pol) {
  if constexpr (kHint)
    asm volatile(
        "st.global.L1::no_allocate.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p),
        "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "l"(pol)
        : "memory");
  else
    asm volatile("st.global.L1::no_allocate.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p),
                 "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t smem, const float *gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem),
               "l"(gmem)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float4 lds128(uint32_t smem) {
  float4 r;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "r"(smem));
  return r;
}

// Byte offset of (row j of lane p, half h) inside a 4 KB stage.  Row
// r = 8p + j is 32 bytes (two 16-byte halves); the 32-byte slot inside each
// 128-byte line is XOR-ed with p & 3 so that the eight lanes of a quarter
// warp (p = 4q..4q+3, h = 0, 1) address eight different 16-byte groups.
__device__ __forceinline__ uint32_t stage_off(int p, int h, int j) {
  const int r = 8 * p + j;
  const int slot = (r & 3) ^ (p & 3);
  return (uint32_t)((r >> 2) * 128 + slot * 32 + h * 16);
}

__device__ __forceinline__ float comp(const float4 &a, int i) {
  return i == 0 ? a.x : (i == 1 ? a.y : (i == 2 ? a.z : a.w));
}

// The per-token inputs a lane needs: k and q for its 8 key rows, v for its 4
// value columns, and the head's two scalars.
struct TokenIn {
  float4 k0, k1, q0, q1, v;
  float g, beta;
};

__device__ __forceinline__ TokenIn load_token(const float *__restrict__ q,
                                              const float *__restrict__ k,
                                              const float *__restrict__ v,
                                              const float *__restrict__ g,
                                              const float *__restrict__ beta,
                                              size_t qk_row, size_t v_row,
                                              size_t gi) {
  TokenIn t;
  const float4 *kp = reinterpret_cast<const float4 *>(k + qk_row);
  const float4 *qp = reinterpret_cast<const float4 *>(q + qk_row);
  t.k0 = __ldg(kp);
  t.k1 = __ldg(kp + 1);
  t.q0 = __ldg(qp);
  t.q1 = __ldg(qp + 1);
  t.v = __ldg(reinterpret_cast<const float4 *>(v + v_row));
  t.g = __ldg(g + gi);
  t.beta = __ldg(beta + gi);
  return t;
}

__device__ __forceinline__ float row_of(const TokenIn &t, bool isq, int j) {
  const float4 &a = isq ? (j < 4 ? t.q0 : t.q1) : (j < 4 ? t.k0 : t.k1);
  return comp(a, j & 3);
}

// Partial dot products of the lane's 8 rows with x (k or q), per column.
__device__ __forceinline__ float4 partial_dot(const float4 (&s)[8],
                                              const TokenIn &t, bool isq) {
  const float x0 = row_of(t, isq, 0);
  float4 a = make_float4(__fmul_rn(s[0].x, x0), __fmul_rn(s[0].y, x0),
                         __fmul_rn(s[0].z, x0), __fmul_rn(s[0].w, x0));
#pragma unroll
  for (int j = 1; j < 8; ++j) {
    const float xj = row_of(t, isq, j);
    a.x = __fmaf_rn(s[j].x, xj, a.x);
    a.y = __fmaf_rn(s[j].y, xj, a.y);
    a.z = __fmaf_rn(s[j].z, xj, a.z);
    a.w = __fmaf_rn(s[j].w, xj, a.w);
  }
  return a;
}

// One token for the lane's 8 x 4 block (lane = 2p + h).  Updates s in place
// and, on the lanes that own an output element, writes it to o_half[c]
// (c = 0..3 is the column inside the lane's 4-column half).
__device__ __forceinline__ void token_update(float4 (&s)[8], const TokenIn &t,
                                             int lane, float *o_half) {
  const int p = lane >> 1;
  const int h = lane & 1;

  // 1. Partials over this lane's rows: S^T k and S^T q for 4 columns, q.k.
  const float4 kv = partial_dot(s, t, false);
  const float4 qs = partial_dot(s, t, true);
  float qk = __fmul_rn(t.q0.x, t.k0.x);
  qk = __fmaf_rn(t.q0.y, t.k0.y, qk);
  qk = __fmaf_rn(t.q0.z, t.k0.z, qk);
  qk = __fmaf_rn(t.q0.w, t.k0.w, qk);
  qk = __fmaf_rn(t.q1.x, t.k1.x, qk);
  qk = __fmaf_rn(t.q1.y, t.k1.y, qk);
  qk = __fmaf_rn(t.q1.z, t.k1.z, qk);
  qk = __fmaf_rn(t.q1.w, t.k1.w, qk);

  // 2. Reduce-scatter the 8 column partials over the 16 lanes sharing h.
  // The 16 row blocks combine in the fixed tree of the file header: p bits
  // 2, 1, 8, 4 in turn (lane xor 4, 2, 16, 8).  Afterwards the lane
  // holds the full sum of value index idx = 4*[p&2] + 2*[p&1] + [p&8]:
  // idx < 4 is S^T k of column idx, idx >= 4 is S^T q of column idx - 4.
  const bool s2 = p & 2, s1 = p & 1, s8 = p & 8;
  float r4[4];
  {
    const float keep[4] = {s2 ? qs.x : kv.x, s2 ? qs.y : kv.y,
                           s2 ? qs.z : kv.z, s2 ? qs.w : kv.w};
    const float send[4] = {s2 ? kv.x : qs.x, s2 ? kv.y : qs.y,
                           s2 ? kv.z : qs.z, s2 ? kv.w : qs.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      r4[i] = __fadd_rn(keep[i], __shfl_xor_sync(kFull, send[i], 4));
  }
  float r2[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = s1 ? r4[i + 2] : r4[i];
    const float send = s1 ? r4[i] : r4[i + 2];
    r2[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, 2));
  }
  float r1;
  {
    const float keep = s8 ? r2[1] : r2[0];
    const float send = s8 ? r2[0] : r2[1];
    r1 = __fadd_rn(keep, __shfl_xor_sync(kFull, send, 16));
  }
  const float red = __fadd_rn(r1, __shfl_xor_sync(kFull, r1, 8));
  const int idx = (s2 ? 4 : 0) + (s1 ? 2 : 0) + (s8 ? 1 : 0);

  // q . k over all 128 rows (the 16 lanes of either half hold every row),
  // in the same tree.
  qk = __fadd_rn(qk, __shfl_xor_sync(kFull, qk, 4));
  qk = __fadd_rn(qk, __shfl_xor_sync(kFull, qk, 2));
  qk = __fadd_rn(qk, __shfl_xor_sync(kFull, qk, 16));
  qk = __fadd_rn(qk, __shfl_xor_sync(kFull, qk, 8));

  // 3. tmp = (v - alpha kv) beta on the S^T k lanes, then broadcast the four
  // columns' tmp to every lane of the same h.  Column c's S^T k lives on
  // p = (c>>1) + 8*(c&1) (and p + 4).
  const float alpha = expf(t.g);
  const int col = idx & 3;
  const float tmp_mine =
      __fmul_rn(__fsub_rn(comp(t.v, col), __fmul_rn(alpha, red)), t.beta);
  float tmp[4];
#pragma unroll
  for (int c = 0; c < 4; ++c)
    tmp[c] = __shfl_sync(kFull, tmp_mine,
                         (((c >> 1) + 8 * (c & 1)) << 1) | h);

  // 4. o = alpha (S^T q) + (q . k) tmp on the S^T q lanes (p & 4 clear:
  // one of the two lanes that hold each sum).
  if (idx >= 4 && !(p & 4)) {
    float tc = tmp[0];
#pragma unroll
    for (int c = 1; c < 4; ++c)
      if (col == c) tc = tmp[c];
    o_half[col] = __fmaf_rn(qk, tc, __fmul_rn(alpha, red));
  }

  // 5. Rank-1 update of the decayed state: S = alpha S + k tmp^T.
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float kj = row_of(t, false, j);
    s[j].x = __fmaf_rn(kj, tmp[0], __fmul_rn(alpha, s[j].x));
    s[j].y = __fmaf_rn(kj, tmp[1], __fmul_rn(alpha, s[j].y));
    s[j].z = __fmaf_rn(kj, tmp[2], __fmul_rn(alpha, s[j].z));
    s[j].w = __fmaf_rn(kj, tmp[3], __fmul_rn(alpha, s[j].w));
  }
}

// Start the copy of unit u's 4 KB into the stage at smem address `stage`.
__device__ __forceinline__ void issue_unit(const float *S_in, size_t u,
                                           uint32_t stage, int p, int h) {
  const size_t head = u / kUnitsPerHead;
  const int cg = (int)(u % kUnitsPerHead);
  const float *src = S_in + head * (size_t)(kDim * kDim) +
                     (size_t)(8 * p) * kDim + 8 * cg + 4 * h;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    cp_async16(stage + stage_off(p, h, j), src + j * kDim);
}

// kOne: launches of one token (decode), whose addressing finds each unit's
// coordinates where its inputs are loaded (measured 0.8 % faster for M = 1);
// otherwise a unit's offsets are found once and stepped per token (5 % faster
// for M = 8).  The arithmetic is the same, so results are the same bits.
template <bool kCkpt, bool kOne, int kWarps>
__global__ void __launch_bounds__(kWarps * 32, kWarpsPerSm / kWarps)
    gdn_steps_kernel(const float *S_in, float *S_out,
                     float *__restrict__ ckpt, const float *__restrict__ q,
                     const float *__restrict__ k, const float *__restrict__ v,
                     const float *__restrict__ g,
                     const float *__restrict__ beta, float *__restrict__ o,
                     int vh, int kh, int rep, int M, size_t nheads,
                     int wait_first) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int p = lane >> 1;
  const int h = lane & 1;
  const uint32_t ring =
      (uint32_t)__cvta_generic_to_shared(smem_raw) +
      (uint32_t)(warp * kStages * kUnitFloats * 4);

  const size_t nunits = nheads * kUnitsPerHead;
  const size_t gw = (size_t)blockIdx.x * kWarps + warp;
  const size_t nw = (size_t)gridDim.x * kWarps;
  const size_t mine = gw < nunits ? (nunits - gw + nw - 1) / nw : 0;
  const uint64_t pol = kOne ? l2_keep_priority() : 0;
  // behind a kernel that may write the state, nothing is read before it ends
  if (wait_first) asm volatile("griddepcontrol.wait;" ::: "memory");

  // Prologue: the first kStages - 1 units in flight (empty groups keep the
  // group count uniform).
#pragma unroll
  for (int st = 0; st < kStages - 1; ++st) {
    if ((size_t)st < mine)
      issue_unit(S_in, gw + st * nw, ring + st * kUnitFloats * 4, p, h);
    cp_async_commit();
  }

  // Token inputs are prefetched one token ahead along the flattened list of
  // (unit, token) items, so the next unit's first token is in flight while
  // the current unit computes.
  auto unit_coords = [&](size_t i, int &b, int &vi, int &hh, int &cg,
                         size_t &head) {
    const size_t u = gw + i * nw;
    head = u / kUnitsPerHead;
    cg = (int)(u % kUnitsPerHead);
    b = (int)(head / vh);
    vi = (int)(head % vh);
    hh = vi / rep;
  };
  auto token_at_one = [&](size_t i) {
    int b, vi, hh, cg;
    size_t head;
    unit_coords(i, b, vi, hh, cg, head);
    const size_t bm = (size_t)b;
    return load_token(q, k, v, g, beta, (bm * kh + hh) * kDim + 8 * p,
                      (bm * vh + vi) * kDim + 8 * cg + 4 * h, bm * vh + vi);
  };
  // M > 1: a unit's offsets of token 0 in q/k and in v/o (same layout) are
  // found once per unit, with the divisions by the head counts (32-bit: the
  // head count is bounded by the state's size); token m adds m times the
  // per-token strides.
  struct UnitAt {
    size_t qk, v;
  };
  auto unit_at = [&](size_t i) {
    const size_t u = gw + i * nw;
    const size_t head = u / kUnitsPerHead;
    const int cg = (int)(u % kUnitsPerHead);
    const unsigned hd32 = (unsigned)head;
    const unsigned b32 = hd32 / (unsigned)vh;
    const int vi = (int)(hd32 - b32 * (unsigned)vh);
    const int hh = vi / rep;
    const size_t bm = (size_t)b32 * (size_t)M;
    return UnitAt{(bm * kh + hh) * kDim + 8 * p,
                  (bm * vh + vi) * kDim + 8 * cg + 4 * h};
  };
  const size_t dqk = (size_t)kh * kDim, dv = (size_t)vh * kDim;
  auto token_at = [&](const UnitAt &a, int m) {
    const size_t vo = a.v + (size_t)m * dv;
    return load_token(q, k, v, g, beta, a.qk + (size_t)m * dqk, vo,
                      vo / kDim);  // (v row) / kDim = (b, token, head) index
  };

  // the token inputs may come from the kernel this one overlaps with
  asm volatile("griddepcontrol.wait;" ::: "memory");
  TokenIn cur;
  UnitAt cu{0, 0}, nu{0, 0};
  if (mine > 0) {
    if constexpr (kOne) {
      cur = token_at_one(0);
    } else {
      cu = unit_at(0);
      cur = token_at(cu, 0);
    }
  }
  for (size_t i = 0; i < mine; ++i) {
    // dependents may be scheduled once every warp is on its last unit
    if (i + 1 == mine) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    {
      const size_t ahead = i + kStages - 1;
      if (ahead < mine)
        issue_unit(S_in, gw + ahead * nw,
                   ring + (uint32_t)(ahead % kStages) * kUnitFloats * 4, p, h);
      cp_async_commit();
    }
    cp_async_wait<kStages - 1>();  // unit i has landed (this lane's bytes)

    const size_t u = gw + i * nw;
    size_t head = u / kUnitsPerHead;
    int col0 = 8 * (int)(u % kUnitsPerHead) + 4 * h;
    size_t o_off = 0;
    if constexpr (kOne) {
      int b, vi, hh, cg;
      unit_coords(i, b, vi, hh, cg, head);
      col0 = 8 * cg + 4 * h;
      o_off = ((size_t)b * vh + vi) * kDim + col0;
    }
    const uint32_t stage = ring + (uint32_t)(i % kStages) * kUnitFloats * 4;

    float4 s[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j] = lds128(stage + stage_off(p, h, j));

    const size_t hoff = head * (size_t)(kDim * kDim);
    const size_t eoff = (size_t)(8 * p) * kDim + col0;
    if constexpr (!kOne && !kCkpt) {
      // tokens in pairs: cur and nxt take turns as the token being computed
      // and the one being loaded, so no inputs are copied between registers
      // (one copy per unit when M is odd)
      TokenIn nxt;
      auto load_after = [&](int m, TokenIn &dst) {
        if (m + 1 < M) {
          dst = token_at(cu, m + 1);
        } else if (i + 1 < mine) {
          nu = unit_at(i + 1);
          dst = token_at(nu, 0);
        }
      };
      for (int m = 0; m < M; m += 2) {
        load_after(m, nxt);
        token_update(s, cur, lane, o + cu.v + (size_t)m * dv);
        if (m + 1 == M) {
          cur = nxt;
          break;
        }
        load_after(m + 1, cur);
        token_update(s, nxt, lane, o + cu.v + (size_t)(m + 1) * dv);
      }
    } else {
      for (int m = 0; m < M; ++m) {
        TokenIn nxt = cur;
        if constexpr (kOne) {
          if (i + 1 < mine) nxt = token_at_one(i + 1);
          token_update(s, cur, lane, o + o_off);
        } else {
          if (m + 1 < M) {
            nxt = token_at(cu, m + 1);
          } else if (i + 1 < mine) {
            nu = unit_at(i + 1);
            nxt = token_at(nu, 0);
          }
          token_update(s, cur, lane, o + cu.v + (size_t)m * dv);
        }
        if (kCkpt) {
          float *cp = ckpt + (size_t)m * nheads * (kDim * kDim) + hoff + eoff;
  #pragma unroll
          for (int j = 0; j < 8; ++j) st_stream<kOne>(cp + j * kDim, s[j], pol);
        }
        cur = nxt;
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) st_stream<kOne>(S_out + hoff + eoff + j * kDim, s[j], pol);
    cu = nu;
  }
  cp_async_wait<0>();
}

// Single-token update with the 32-column layout (see the file header).  A
// unit is (head, 32-column group cg); a CTA of 4 warps walks a strided list
// of units.  Warp w holds key rows 32w .. 32w+31 of the unit's 32 columns;
// lane = 8 rq + cq holds rows 32w + 8rq .. +7 (block p = 4w + rq) of columns
// 32cg + 4cq .. +3.  Each warp keeps its next kStages - 1 quarter-units in
// flight with cp.async into a private ring (a lane reads back only what it
// copied).  Per unit each lane reduces its block's partials over rq inside
// the warp (rq bit 1, then bit 0: the first two levels of the tree), writes
// them to an exchange buffer (by unit parity), and after one CTA barrier
// every lane finishes S^T k for its 4 columns over the 4 warps, (W_0 + W_2)
// + (W_1 + W_3); warp 0's lanes 0-7 also finish S^T q and write o.  The
// arithmetic is token_update's, term for term.
constexpr int kC32Warps = 4;                          // warps per column group
// Column groups per CTA when the token inputs are in host memory: 2 (a
// 64 x 48-head step took 67.9 us end to end, against 78.8 us with 4 groups,
// whose 16-warp CTAs run one per SM and wait longer at their barrier, and
// 70.1 us for the 8-column layout with 8-warp CTAs).
constexpr int kHostGroups = 2;
constexpr int kC32Groups = kDim / 32;                 // column groups per head
constexpr int kC32Stage = 32 * 32 * 4;                // one warp's 4 KB
template <int G>
__host__ __device__ constexpr int c32_smem() {
  return G * kC32Warps * kStages * kC32Stage + G * (2 * kC32Warps * 64 + 2 * kC32Warps) * 4;
}

// G column groups of a head per CTA (4 G warps): G = 1 for device-resident
// inputs; G = kHostGroups when the token inputs are in host memory, so that
// the CTA's column groups share a head's q and k rows in L1 and the rows
// cross the host link fewer times.
template <int G, bool kWaitFirst>
__global__ void __launch_bounds__(G * kC32Warps * 32, kWarpsPerSm / (G * kC32Warps))
    gdn_step_c32_kernel(const float *S_in, float *S_out,
                        const float *__restrict__ q,
                        const float *__restrict__ k,
                        const float *__restrict__ v,
                        const float *__restrict__ g,
                        const float *__restrict__ beta,
                        float *__restrict__ o, int vh, int kh, int rep,
                        size_t nheads) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int warp = wid & (kC32Warps - 1), grp = wid / kC32Warps;
  const int rq = lane >> 3, cq = lane & 7;
  const uint32_t ring = (uint32_t)__cvta_generic_to_shared(smem_raw) +
                        (uint32_t)(wid * kStages * kC32Stage);
  // exchange per group: [parity][warp][cq][kv0..3, qs0..3] and
  // [parity][warp] q . k
  float *xch = reinterpret_cast<float *>(smem_raw + G * kC32Warps * kStages * kC32Stage) +
               grp * (2 * kC32Warps * 64 + 2 * kC32Warps);
  float *qkx = xch + 2 * kC32Warps * 64;
  const size_t nunits = nheads * (kC32Groups / G);
  const size_t mine =
      blockIdx.x < nunits ? (nunits - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const uint64_t pol = l2_keep_priority();
  const int r0 = 32 * warp + 8 * rq;
  const uint32_t lane_off = (uint32_t)(8 * rq * 128 + cq * 16);
  // behind a kernel that may write the state, nothing is read before it ends
  if constexpr (kWaitFirst) asm volatile("griddepcontrol.wait;" ::: "memory");

  auto issue = [&](size_t i, int st) {
    const size_t u = blockIdx.x + i * gridDim.x;
    const size_t head = u / (kC32Groups / G);
    const int cg = (int)(u % (kC32Groups / G)) * G + grp;
    const float *src = S_in + head * (size_t)(kDim * kDim) + (size_t)r0 * kDim +
                       32 * cg + 4 * cq;
    const uint32_t dst = ring + (uint32_t)(st * kC32Stage) + lane_off;
#pragma unroll
    for (int j = 0; j < 8; ++j) cp_async16(dst + j * 128, src + j * kDim);
  };
#pragma unroll
  for (int st = 0; st < kStages - 1; ++st) {
    if ((size_t)st < mine) issue(st, st);
    cp_async_commit();
  }
  // the token inputs may come from the kernel this one overlaps with
  if constexpr (!kWaitFirst) asm volatile("griddepcontrol.wait;" ::: "memory");

  for (size_t i = 0; i < mine; ++i) {
    // dependents may be scheduled once every CTA is on its last unit: a
    // following step's CTAs then take the slots as these CTAs leave, and
    // small CTAs of another kernel do not wait beside this one's for long
    if (i + 1 == mine) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    {
      const size_t ahead = i + kStages - 1;
      if (ahead < mine) issue(ahead, (int)(ahead % kStages));
      cp_async_commit();
    }
    const size_t u = blockIdx.x + i * gridDim.x;
    const size_t head = u / (kC32Groups / G);
    const int cg = (int)(u % (kC32Groups / G)) * G + grp;
    const int b = (int)(head / vh), vi = (int)(head % vh), hh = vi / rep;
    const TokenIn t = load_token(q, k, v, g, beta, ((size_t)b * kh + hh) * kDim + r0,
                                 ((size_t)b * vh + vi) * kDim + 32 * cg + 4 * cq,
                                 (size_t)b * vh + vi);
    cp_async_wait<kStages - 1>();  // unit i has landed (this lane's bytes)
    const uint32_t stage = ring + (uint32_t)((i % kStages) * kC32Stage) + lane_off;
    float4 s[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j] = lds128(stage + j * 128);

    // partials over this lane's 8 rows, as in token_update
    const float4 kv = partial_dot(s, t, false);
    const float4 qs = partial_dot(s, t, true);
    float qk = __fmul_rn(t.q0.x, t.k0.x);
    qk = __fmaf_rn(t.q0.y, t.k0.y, qk);
    qk = __fmaf_rn(t.q0.z, t.k0.z, qk);
    qk = __fmaf_rn(t.q0.w, t.k0.w, qk);
    qk = __fmaf_rn(t.q1.x, t.k1.x, qk);
    qk = __fmaf_rn(t.q1.y, t.k1.y, qk);
    qk = __fmaf_rn(t.q1.z, t.k1.z, qk);
    qk = __fmaf_rn(t.q1.w, t.k1.w, qk);

    // tree levels 1 and 2 inside the warp: rq bit 1 (lane xor 16), then
    // rq bit 0 (lane xor 8); the lane keeps 2 of its 8 values: kv or qs by
    // rq bit 1, columns (0, 1) or (2, 3) by rq bit 0
    const bool t1 = rq & 2, t0 = rq & 1;
    float r4[4];
    {
      const float keep[4] = {t1 ? qs.x : kv.x, t1 ? qs.y : kv.y,
                             t1 ? qs.z : kv.z, t1 ? qs.w : kv.w};
      const float send[4] = {t1 ? kv.x : qs.x, t1 ? kv.y : qs.y,
                             t1 ? kv.z : qs.z, t1 ? kv.w : qs.w};
#pragma unroll
      for (int c = 0; c < 4; ++c)
        r4[c] = __fadd_rn(keep[c], __shfl_xor_sync(kFull, send[c], 16));
    }
    float r2[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const float keep = t0 ? r4[c + 2] : r4[c];
      const float send = t0 ? r4[c] : r4[c + 2];
      r2[c] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, 8));
    }
    qk = __fadd_rn(qk, __shfl_xor_sync(kFull, qk, 16));
    qk = __fadd_rn(qk, __shfl_xor_sync(kFull, qk, 8));

    const int par = (int)(i & 1);
    float *X = xch + par * (kC32Warps * 64);
    *reinterpret_cast<float2 *>(X + warp * 64 + cq * 8 + rq * 2) =
        make_float2(r2[0], r2[1]);
    if (lane == 0) qkx[par * kC32Warps + warp] = qk;
    __syncthreads();  // the exchange of unit i is complete

    // tree levels 3 and 4 across the warps: (W_0 + W_2) + (W_1 + W_3)
    auto across = [&](int off) {
      const float4 w0 = *reinterpret_cast<const float4 *>(X + 0 * 64 + cq * 8 + off);
      const float4 w1 = *reinterpret_cast<const float4 *>(X + 1 * 64 + cq * 8 + off);
      const float4 w2 = *reinterpret_cast<const float4 *>(X + 2 * 64 + cq * 8 + off);
      const float4 w3 = *reinterpret_cast<const float4 *>(X + 3 * 64 + cq * 8 + off);
      return make_float4(__fadd_rn(__fadd_rn(w0.x, w2.x), __fadd_rn(w1.x, w3.x)),
                         __fadd_rn(__fadd_rn(w0.y, w2.y), __fadd_rn(w1.y, w3.y)),
                         __fadd_rn(__fadd_rn(w0.z, w2.z), __fadd_rn(w1.z, w3.z)),
                         __fadd_rn(__fadd_rn(w0.w, w2.w), __fadd_rn(w1.w, w3.w)));
    };
    const float4 kvs = across(0);
    const float* Q = qkx + par * kC32Warps;
    const float qkt = __fadd_rn(__fadd_rn(Q[0], Q[2]), __fadd_rn(Q[1], Q[3]));
    const float alpha = expf(t.g);
    float tmp[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
      tmp[c] = __fmul_rn(__fsub_rn(comp(t.v, c), __fmul_rn(alpha, comp(kvs, c))),
                         t.beta);
    if (warp == 0 && rq == 0) {
      const float4 qss = across(4);
      float4 ov;
      ov.x = __fmaf_rn(qkt, tmp[0], __fmul_rn(alpha, qss.x));
      ov.y = __fmaf_rn(qkt, tmp[1], __fmul_rn(alpha, qss.y));
      ov.z = __fmaf_rn(qkt, tmp[2], __fmul_rn(alpha, qss.z));
      ov.w = __fmaf_rn(qkt, tmp[3], __fmul_rn(alpha, qss.w));
      *reinterpret_cast<float4 *>(o + ((size_t)b * vh + vi) * kDim + 32 * cg + 4 * cq) = ov;
    }
    // S = alpha S + k tmp^T
    float *dst = S_out + head * (size_t)(kDim * kDim) + (size_t)r0 * kDim + 32 * cg + 4 * cq;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float kj = row_of(t, false, j);
      float4 n;
      n.x = __fmaf_rn(kj, tmp[0], __fmul_rn(alpha, s[j].x));
      n.y = __fmaf_rn(kj, tmp[1], __fmul_rn(alpha, s[j].y));
      n.z = __fmaf_rn(kj, tmp[2], __fmul_rn(alpha, s[j].z));
      n.w = __fmaf_rn(kj, tmp[3], __fmul_rn(alpha, s[j].w));
      st_stream<true>(dst + j * kDim, n, pol);
    }
  }
  cp_async_wait<0>();
}

// Multi-token update (M > 1, no checkpoints) with device-resident token
// inputs: one CTA of 8 warps per head, warp c on the head's 16-column group
// c.  Lane = 4 rg + cq holds columns 16 c + 4 cq .. +3 of the two 8-row
// blocks that the first level of the reduction tree adds: rg = 2 w + j,
// blocks pA = 4 w + j and pB = pA + 2 (rows 8 pA .. +7 and 8 pB .. +7).  So
// the lane's own partials already form B_pA + B_pB (tree level 1), and the
// remaining levels are lane xor 4 (j: W_w), xor 16 (w bit 1: W_0 + W_2,
// W_1 + W_3) and xor 8 (w bit 0): the tree of the file header term for
// term, so a token gives the same bits here as in the single-token kernels.
// After the reduce-scatter, lane (w, j, cq) holds S^T k (j = 0) or S^T q
// (j = 1) of column 4 cq + w; the j = 0 lanes form tmp, four shuffles give
// every lane its columns' tmp, and the j = 1 lanes write o.  The state
// arithmetic runs as packed pairs (__ffma2_rn / __fmul2_rn: per component
// the rounding of __fmaf_rn / __fmul_rn).
//
// Token inputs.  The head's q, k and v rows of a token (512 bytes each) are
// shared by the CTA's 8 warps through a ring of kHSlots slots in shared
// memory, filled by bulk copies (cp.async.bulk, completion on one mbarrier
// per slot) kHSlots - 1 tokens ahead: the warp that releases a slot last
// (a shared counter) refills it with the token kHSlots further on, so no
// warp waits for another except through the ring itself.  g and beta come
// 32 tokens at a time, one token per lane (loaded a chunk ahead), alpha =
// exp(g) computed once per token, and reach every lane by shuffles.  With
// q, k and v read from shared memory as they are used, no token input is
// held in registers across a token.
//
// State.  Each warp copies its next unit's 8 KB with cp.async into a private
// stage as soon as it has read the current one into registers, so one unit
// is in flight while one computes; a lane reads back only what it copied.
// The stage layout [register r][lane] makes every 128-bit shared access of a
// quarter warp one contiguous 128-byte line; the q and k reads of a quarter
// warp touch two addresses (broadcast), so no access has bank conflicts.
//
// Waits on the ring are bounded: a wait that runs out counts a time-out
// (gdn_wait_timeouts), marks every result the CTA had not yet written as NaN
// (state and o of the remaining units), and the CTA waits, bounded again,
// for its copies in flight before it exits.
constexpr int kHWarps = 8;
constexpr int kHCtasPerSm = 2;
constexpr int kHSlots = 6;
constexpr int kHStage = 16 * kDim * 4;                   // one warp's 8 KB
constexpr int kHSlotBytes = 3 * kDim * 4;                // k | q | v rows
constexpr int kHOffSlots = kHWarps * kHStage;
constexpr int kHOffBar = kHOffSlots + kHSlots * kHSlotBytes;
constexpr int kHOffCnt = kHOffBar + kHSlots * 8;
constexpr int kHOffLast = kHOffCnt + kHSlots * 4;
constexpr int kHOffFail = kHOffLast + kHSlots * 4;
constexpr int kHSmem = kHOffFail + 16;
constexpr uint32_t kHWaitLimit = 1u << 24;

__device__ unsigned int g_steps_timeouts = 0;

__device__ __forceinline__ float4 f4_of(float2 lo, float2 hi) {
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}

// sum over the 8 rows of a block (row order) of s[row] * x[row]: the first
// product rounded, then fused multiply-adds -- partial_dot's arithmetic.
__device__ __forceinline__ float4 block_dot(const float4 *s, const float4 &x0,
                                            const float4 &x1) {
  float2 lo = __fmul2_rn(make_float2(s[0].x, s[0].y), make_float2(x0.x, x0.x));
  float2 hi = __fmul2_rn(make_float2(s[0].z, s[0].w), make_float2(x0.x, x0.x));
#pragma unroll
  for (int r = 1; r < 8; ++r) {
    const float xr = comp(r < 4 ? x0 : x1, r & 3);
    const float2 xx = make_float2(xr, xr);
    lo = __ffma2_rn(make_float2(s[r].x, s[r].y), xx, lo);
    hi = __ffma2_rn(make_float2(s[r].z, s[r].w), xx, hi);
  }
  return f4_of(lo, hi);
}

__device__ __forceinline__ float block_qk(const float4 &q0, const float4 &q1,
                                          const float4 &k0, const float4 &k1) {
  float a = __fmul_rn(q0.x, k0.x);
  a = __fmaf_rn(q0.y, k0.y, a);
  a = __fmaf_rn(q0.z, k0.z, a);
  a = __fmaf_rn(q0.w, k0.w, a);
  a = __fmaf_rn(q1.x, k1.x, a);
  a = __fmaf_rn(q1.y, k1.y, a);
  a = __fmaf_rn(q1.z, k1.z, a);
  a = __fmaf_rn(q1.w, k1.w, a);
  return a;
}

__device__ __forceinline__ float4 add4(const float4 &a, const float4 &b) {
  return f4_of(__fadd2_rn(make_float2(a.x, a.y), make_float2(b.x, b.y)),
               __fadd2_rn(make_float2(a.z, a.w), make_float2(b.z, b.w)));
}

__device__ __forceinline__ void bulk_load(uint32_t smem, const float *src,
                                          uint32_t bytes, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1], %2, [%3];" ::"r"(smem),
      "l"(src), "r"(bytes), "r"(mbar)
      : "memory");
}

__device__ __forceinline__ void arrive_expect_tx(uint32_t mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar),
               "r"(bytes)
               : "memory");
}

// Shared-memory fetch-and-add with acquire-release ordering at CTA scope.
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned *p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ float lds32(uint32_t smem) {
  float r;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(r) : "r"(smem));
  return r;
}

__global__ void __launch_bounds__(kHWarps * 32, kHCtasPerSm)
    gdn_steps_head_kernel(const float *S_in, float *S_out,
                          const float *__restrict__ q,
                          const float *__restrict__ k,
                          const float *__restrict__ v,
                          const float *__restrict__ g,
                          const float *__restrict__ beta,
                          float *__restrict__ o, int vh, int kh, int rep, int M,
                          unsigned nheads, int wait_first) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rg = lane >> 2, cq = lane & 3;
  const int j = rg & 1, w = rg >> 1;
  const int rowA = 8 * (4 * w + j);             // block pA; pB = rows + 16
  const int col = 16 * warp + 4 * cq;           // the lane's first column
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t stage = sbase + (uint32_t)(warp * kHStage + lane * 16);
  const uint32_t slots = sbase + kHOffSlots;
  const uint32_t bars = sbase + kHOffBar;
  unsigned int *cnt = reinterpret_cast<unsigned int *>(smem_raw + kHOffCnt);
  int *last = reinterpret_cast<int *>(smem_raw + kHOffLast);
  int *failed = reinterpret_cast<int *>(smem_raw + kHOffFail);
  const unsigned mine =
      blockIdx.x < nheads ? (nheads - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const size_t hstride = (size_t)vh * kDim;     // o / v stride per token
  // behind a kernel that may write the state, nothing is read before it ends
  if (wait_first) asm volatile("griddepcontrol.wait;" ::: "memory");

  auto head_of = [&](unsigned i) { return blockIdx.x + i * gridDim.x; };
  // offset of this lane's first state element (row rowA, column col) in
  // unit i's head; its 16 rows are at + r * kDim (r < 8) and + (r + 8) * kDim
  auto s_off = [&](unsigned i) {
    return (size_t)head_of(i) * (kDim * kDim) + (size_t)(rowA * kDim + col);
  };
  auto issue_state = [&](unsigned i) {
    const float *src = S_in + s_off(i);
#pragma unroll
    for (int r = 0; r < 16; ++r)
      cp_async16(stage + r * 512, src + (r < 8 ? r : r + 8) * kDim);
  };
  if (mine > 0) issue_state(0);
  cp_async_commit();

  if (threadIdx.x == 0) {
    for (int sl = 0; sl < kHSlots; ++sl) {
      tc::mbar_init(bars + 8 * sl, 1);
      cnt[sl] = 0;
      last[sl] = -1;
    }
    *failed = 0;
  }
  __syncthreads();

  // the k, q and v rows of token m of unit i into slot sl, whose use-th
  // filling this is (one thread at a time)
  auto issue_item = [&](unsigned i, int m, int sl, int use) {
    const unsigned head = head_of(i);
    const unsigned b = head / (unsigned)vh;
    const unsigned vi = head - b * (unsigned)vh;
    const unsigned hh = vi / (unsigned)rep;
    const size_t bm = (size_t)b * (size_t)M + (size_t)m;
    const uint32_t dst = slots + (uint32_t)(sl * kHSlotBytes);
    const uint32_t bar = bars + 8 * sl;
    last[sl] = use;
    tc::fence_proxy_async();
    arrive_expect_tx(bar, kHSlotBytes);
    bulk_load(dst, k + (bm * kh + hh) * kDim, kDim * 4, bar);
    bulk_load(dst + kDim * 4, q + (bm * kh + hh) * kDim, kDim * 4, bar);
    bulk_load(dst + 2 * kDim * 4, v + (bm * vh + vi) * kDim, kDim * 4, bar);
  };
  // (unit, token) kHSlots items after (i, m)
  auto ahead = [&](unsigned &i2, int &m2) {
    m2 += kHSlots;
    while (m2 >= M) {
      m2 -= M;
      ++i2;
    }
  };

  // the token inputs may come from the kernel this one overlaps with
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) {
    unsigned i2 = 0;
    int m2 = 0;
    for (int sl = 0; sl < kHSlots && i2 < mine; ++sl) {
      issue_item(i2, m2, sl, 0);
      if (++m2 == M) {
        m2 = 0;
        ++i2;
      }
    }
  }

  // g and beta of the 32 tokens m0 .. m0 + 31 of unit i, one per lane
  auto gb_load = [&](unsigned i, int m0, float &gv, float &bv) {
    gv = 0.0f;
    bv = 0.0f;
    const int m = m0 + lane;
    if (i < mine && m < M) {
      const unsigned head = head_of(i);
      const unsigned b = head / (unsigned)vh;
      const size_t gi = ((size_t)b * (size_t)M + (size_t)m) * (size_t)vh + (head - b * (unsigned)vh);
      gv = __ldg(g + gi);
      bv = __ldg(beta + gi);
    }
  };
  float g_nx, b_nx, a_ch = 0.0f, b_ch = 0.0f;
  gb_load(0, 0, g_nx, b_nx);

  // j = 1 lanes take q as their first operand and k as their second, so the
  // first reduction level keeps its first vector on every lane
  const uint32_t x1off = (uint32_t)(rowA * 4 + (j ? kDim * 4 : 0));
  const uint32_t x2off = (uint32_t)(rowA * 4 + (j ? 0 : kDim * 4));
  const uint32_t koff = (uint32_t)(rowA * 4);
  const uint32_t voff = (uint32_t)(2 * kDim * 4 + (col + w) * 4);

  float4 s[16];
  bool ok = true;
  unsigned i = 0;
  int m = 0, sl = 0, use = 0;
  for (; i < mine; ++i) {
    // dependents may be scheduled once every CTA is on its last unit
    if (i + 1 == mine) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    cp_async_wait<0>();  // unit i has landed (this lane's bytes)
#pragma unroll
    for (int r = 0; r < 16; ++r) s[r] = lds128(stage + r * 512);
    if (i + 1 < mine) issue_state(i + 1);  // after this lane's own reads
    cp_async_commit();
    const size_t soff = s_off(i);
    float *op;
    {
      const unsigned head = head_of(i);
      const unsigned b = head / (unsigned)vh;
      op = o + ((size_t)b * (size_t)M * vh + (head - b * (unsigned)vh)) * kDim + col + w;
    }

    for (m = 0; m < M; ++m) {
      if ((m & 31) == 0) {  // the next 32 tokens' gates, and the chunk after
        a_ch = expf(g_nx);
        b_ch = b_nx;
        if (m + 32 < M) gb_load(i, m + 32, g_nx, b_nx);
        else gb_load(i + 1, 0, g_nx, b_nx);
      }
      const float alpha = __shfl_sync(kFull, a_ch, m & 31);
      const float bt = __shfl_sync(kFull, b_ch, m & 31);
      const uint32_t slot = slots + (uint32_t)(sl * kHSlotBytes);
      if (!__all_sync(kFull, tc::mbar_wait(bars + 8 * sl, (uint32_t)(use & 1),
                                           kHWaitLimit))) {
        ok = false;
        break;
      }

      // partials of blocks A and B, then tree level 1 (B_pA + B_pB); x1 is
      // k on j = 0 lanes and q on j = 1 lanes
      float4 d1, d2;
      float qk;
      {
        const float4 a0 = lds128(slot + x1off), a1 = lds128(slot + x1off + 16);
        const float4 b0 = lds128(slot + x2off), b1 = lds128(slot + x2off + 16);
        d1 = block_dot(s, a0, a1);
        d2 = block_dot(s, b0, b1);
        qk = block_qk(a0, a1, b0, b1);
      }
      {
        const float4 a0 = lds128(slot + x1off + 64), a1 = lds128(slot + x1off + 80);
        const float4 b0 = lds128(slot + x2off + 64), b1 = lds128(slot + x2off + 80);
        d1 = add4(d1, block_dot(s + 8, a0, a1));
        d2 = add4(d2, block_dot(s + 8, b0, b1));
        qk = __fadd_rn(qk, block_qk(a0, a1, b0, b1));
      }
      // level 2 (lane xor 4): j = 0 keeps S^T k, j = 1 keeps S^T q
      float r4[4];
      r4[0] = __fadd_rn(d1.x, __shfl_xor_sync(kFull, d2.x, 4));
      r4[1] = __fadd_rn(d1.y, __shfl_xor_sync(kFull, d2.y, 4));
      r4[2] = __fadd_rn(d1.z, __shfl_xor_sync(kFull, d2.z, 4));
      r4[3] = __fadd_rn(d1.w, __shfl_xor_sync(kFull, d2.w, 4));
      // level 3 (lane xor 16): w bit 1 keeps columns (2, 3), else (0, 1)
      const bool w1 = w & 2, w0 = w & 1;
      float r2[2];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const float keep = w1 ? r4[c + 2] : r4[c];
        const float send = w1 ? r4[c] : r4[c + 2];
        r2[c] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, 16));
      }
      // level 4 (lane xor 8): w bit 0 keeps the odd column of the pair
      const float red = __fadd_rn(w0 ? r2[1] : r2[0],
                                  __shfl_xor_sync(kFull, w0 ? r2[0] : r2[1], 8));
      qk = __fadd_rn(qk, __shfl_xor_sync(kFull, qk, 4));
      qk = __fadd_rn(qk, __shfl_xor_sync(kFull, qk, 16));
      qk = __fadd_rn(qk, __shfl_xor_sync(kFull, qk, 8));

      // tmp of column col + w on the j = 0 lanes; every lane gets its four
      // columns' tmp from lanes 8 c + cq
      const float vv = lds32(slot + voff);
      const float tmp_mine = __fmul_rn(__fsub_rn(vv, __fmul_rn(alpha, red)), bt);
      float tmp[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmp[c] = __shfl_sync(kFull, tmp_mine, 8 * c + cq);
      const float tmp_pair = __shfl_xor_sync(kFull, tmp_mine, 4);
      if (j)  // o = alpha (S^T q) + (q . k) tmp
        *op = __fmaf_rn(qk, tmp_pair, __fmul_rn(alpha, red));
      op += hstride;

      // S = alpha S + k tmp^T
      {
        const float2 al = make_float2(alpha, alpha);
        const float2 t01 = make_float2(tmp[0], tmp[1]), t23 = make_float2(tmp[2], tmp[3]);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float4 kk4 = lds128(slot + koff + (h < 2 ? 16 * h : 64 + 16 * (h - 2)));
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = 4 * h + e;
            const float kr = comp(kk4, e);
            const float2 kk = make_float2(kr, kr);
            s[r] = f4_of(__ffma2_rn(kk, t01, __fmul2_rn(al, make_float2(s[r].x, s[r].y))),
                         __ffma2_rn(kk, t23, __fmul2_rn(al, make_float2(s[r].z, s[r].w))));
          }
        }
      }
      // release the slot; the warp that releases it last refills it
      __syncwarp();
      if (lane == 0) {
        // release this warp's reads of the slot; the last warp acquires
        // everyone's before it lets the copy engine overwrite the slot
        if ((atom_add_acq_rel(cnt + sl, 1u) & (kHWarps - 1)) == kHWarps - 1) {
          unsigned i2 = i;
          int m2 = m;
          ahead(i2, m2);
          if (i2 < mine) issue_item(i2, m2, sl, use + 1);
        }
      }
      if (++sl == kHSlots) {
        sl = 0;
        ++use;
      }
    }
    if (!ok) break;
    float *dst = S_out + soff;
#pragma unroll
    for (int r = 0; r < 16; ++r) st_stream<false>(dst + (r < 8 ? r : r + 8) * kDim, s[r], 0);
  }

  if (!ok) {
    // a wait ran out: every result of this warp not yet written becomes NaN
    // (the state of unit i on, o of token m of unit i on)
    if (lane == 0 && atomicExch(failed, 1) == 0) atomicAdd(&g_steps_timeouts, 1u);
    const float nan = __int_as_float(0x7fffffff);
    const float4 nan4 = make_float4(nan, nan, nan, nan);
    for (unsigned ii = i; ii < mine; ++ii) {
      const size_t soff = s_off(ii);
      const unsigned head = head_of(ii);
      const unsigned b = head / (unsigned)vh;
      float *op = o + ((size_t)b * (size_t)M * vh + (head - b * (unsigned)vh)) * kDim + col + w;
      for (int r = 0; r < 16; ++r) st_stream<false>(S_out + soff + (r < 8 ? r : r + 8) * kDim, nan4, 0);
      if (j)
        for (int mm = ii == i ? m : 0; mm < M; ++mm) op[(size_t)mm * hstride] = nan;
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  // copies still in flight into the ring (only after a time-out): wait for
  // them, bounded, before the CTA's shared memory is released
  if (threadIdx.x == 0 && *failed)
    for (int q_ = 0; q_ < kHSlots; ++q_)
      if (last[q_] >= 0)
        tc::mbar_wait(bars + 8 * q_, (uint32_t)(last[q_] & 1), kHWaitLimit);
}

// One tile of kCopyUnroll x blockDim 16-byte elements per CTA, as many CTAs
// as tiles: a thread has its kCopyUnroll loads in flight before it stores,
// and the hardware hands tiles to SMs as they free up.  For the 201 MB state
// this measured 61.0 us against 64.9 us for a grid-stride loop over 16 CTAs
// per SM with one load in flight.
constexpr int kCopyUnroll = 4;

__global__ void copy_kernel(float4 *__restrict__ dst,
                            const float4 *__restrict__ src, size_t n4) {
  const size_t base = (size_t)blockIdx.x * blockDim.x * kCopyUnroll;
  float4 r[kCopyUnroll];
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) {
    const size_t i = base + (size_t)u * blockDim.x + threadIdx.x;
    if (i < n4) r[u] = __ldg(src + i);
  }
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) {
    const size_t i = base + (size_t)u * blockDim.x + threadIdx.x;
    if (i < n4) dst[i] = r[u];
  }
}

// One CTA per tile of a (b, vi) head (kRollTiles tiles of 256 threads x
// kCopyUnroll 16-byte elements): copies that tile of the source the
// sequence's count selects, with all of a thread's loads in flight before
// its stores, as copy_kernel does (64 x 48 heads after an 8-token verify:
// 0.935 of the measured copy rate with one CTA per head and a load-store
// loop).
constexpr int kRollTiles = kDim * kDim / 4 / (256 * kCopyUnroll);
static_assert(kRollTiles * 256 * kCopyUnroll == kDim * kDim / 4,
              "a head is a whole number of tiles");
__global__ void rollback_seq_kernel(float4 *__restrict__ S,
                                    const float4 *__restrict__ snap,
                                    const float4 *__restrict__ ckpt,
                                    const int *__restrict__ m_dev,
                                    int *__restrict__ err, int vh, int M,
                                    size_t nheads) {
  const size_t head = blockIdx.x / kRollTiles;
  const int tile = (int)(blockIdx.x % kRollTiles);
  const int b = static_cast<int>(head / vh);
  const int m = __ldg(m_dev + b);
  constexpr size_t n4 = kDim * kDim / 4;
  if (m < 0 || m > M) {
    if (err && threadIdx.x == 0) *err = 1;
    return;
  }
  const size_t off = head * n4 + (size_t)tile * (256 * kCopyUnroll) + threadIdx.x;
  const float4 *src = m == 0 ? snap + off
                             : ckpt + (size_t)(m - 1) * nheads * n4 + off;
  float4 r[kCopyUnroll];
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) r[u] = __ldg(src + u * 256);
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) S[off + u * 256] = r[u];
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
          cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 152;
  }
  return n;
}

}  // namespace

// Launch with the programmatic-dependent attribute when `overlap` is set.
template <typename... Params, typename... Args>
cudaError_t launch_maybe_overlapped(void (*kernel)(Params...), dim3 grid,
                                    dim3 block, size_t smem,
                                    cudaStream_t stream, bool overlap,
                                    Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_steps(const float *S_in, float *S_out, float *ckpt,
                         const float *q, const float *k, const float *v,
                         const float *g, const float *beta, float *o, int B,
                         int kh, int vh, int M, cudaStream_t stream,
                         int overlap, bool host_inputs) {
  const size_t nheads = (size_t)B * vh;
  const size_t nunits = nheads * kUnitsPerHead;
  if (nunits == 0) return cudaSuccess;
  // Behind any kernel only for short launches without checkpoints.  A long
  // launch gains nothing from an earlier start, and its CTAs would wait on
  // SM slots beside the previous launch's last CTAs (8 x 48 heads, 4096
  // tokens: 7.37 ms against 6.75 ms).  Checkpointing launches, bound by
  // their stores, measured mixed (64 x 48 heads, M = 4: 195.2 against
  // 192.6 us; 32 x 48 heads, M = 2: 65.9 against 67.5 us).
  if (overlap == kOverlapAny && (M > kOverlapMaxTokens || ckpt))
    overlap = kOverlapNone;
  if (M == 1 && !ckpt) {
    // one token: the 32-column layout, G column groups of a head per CTA
    auto go32 = [&](auto kernel, int G) {
      const size_t units = nheads * (kC32Groups / G);
      size_t ctas = (size_t)sm_count() * (kWarpsPerSm / (G * kC32Warps));
      if (ctas > units) ctas = units;
      const int smem = G == 1 ? c32_smem<1>() : G == 2 ? c32_smem<2>() : c32_smem<4>();
      const cudaError_t e = cudaFuncSetAttribute(
          kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      return launch_maybe_overlapped(kernel, dim3((unsigned)ctas),
                                     dim3(G * kC32Warps * 32), smem, stream,
                                     overlap, S_in, S_out, q, k, v, g, beta, o,
                                     vh, kh, vh / kh, nheads);
    };
    static_assert(kHostGroups == 2, "host-input launches use two groups");
    const int G = host_inputs ? kHostGroups : 1;
    // Behind any kernel only when the grid fills every CTA slot.  There
    // the launch and the start of the CTAs overlap the previous kernel's
    // end: 64 x 48 heads, 62.8 us against 65.0 us.  A smaller launch (one
    // sequence of 48 heads, state in L2) loses more by loading its state
    // only after the wait: 2.83 us against 2.65 us a step from a graph.
    const bool full = nheads * (kC32Groups / G) >=
                      (size_t)sm_count() * (kWarpsPerSm / (G * kC32Warps));
    if (overlap == kOverlapAny && !full) overlap = kOverlapNone;
    if (overlap == kOverlapAny)
      return host_inputs ? go32(gdn_step_c32_kernel<kHostGroups, true>, kHostGroups)
                         : go32(gdn_step_c32_kernel<1, true>, 1);
    return host_inputs ? go32(gdn_step_c32_kernel<kHostGroups, false>, kHostGroups)
                       : go32(gdn_step_c32_kernel<1, false>, 1);
  }
  const size_t sms = (size_t)sm_count();
  if (!host_inputs && !ckpt && nheads >= sms) {
    // several tokens, device-resident inputs, no checkpoints, at least one
    // head per SM: one CTA per head (head indices in 32 bits).  Fewer heads
    // spread better over the SMs in the 8-column layout (one sequence of
    // 48 heads, 64 tokens: 41 us there against 56 us here), and
    // checkpointing launches, bound by their stores, ran faster there too
    // (64 x 48 heads, M = 2 / 4 / 8: 136 / 194 / 326 us against 139 / 213 /
    // 355 us here).
    if (nheads > 0xffffffffull) return cudaErrorInvalidConfiguration;
    size_t ctas = sms * kHCtasPerSm;
    if (ctas > nheads) ctas = nheads;
    // behind any kernel only when the grid fills every CTA slot (as for
    // one token)
    if (overlap == kOverlapAny && ctas < sms * kHCtasPerSm) overlap = kOverlapNone;
    const cudaError_t e = cudaFuncSetAttribute(
        gdn_steps_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kHSmem);
    if (e != cudaSuccess) return e;
    return launch_maybe_overlapped(gdn_steps_head_kernel, dim3((unsigned)ctas),
                                   dim3(kHWarps * 32), kHSmem, stream, overlap,
                                   S_in, S_out, q, k, v, g, beta, o, vh, kh,
                                   vh / kh, M, (unsigned)nheads,
                                   (int)(overlap == kOverlapAny));
  }
  const int wpc = M == 1 && host_inputs ? 8 : 4;
  const int smem = wpc == 8 ? smem_per_cta<8>() : smem_per_cta<4>();
  size_t ctas = (nunits + wpc - 1) / wpc;
  const size_t cap = sms * (kWarpsPerSm / wpc);
  if (ctas > cap) ctas = cap;
  if (overlap == kOverlapAny && ctas < cap) overlap = kOverlapNone;
  const int wait_first = overlap == kOverlapAny;
  const dim3 grid((unsigned)ctas), block(wpc * 32);
  auto go = [&](auto kernel, float *ck) {
    cudaError_t e = cudaFuncSetAttribute(
        kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_maybe_overlapped(kernel, grid, block, smem, stream,
                                   overlap, S_in, S_out, ck, q, k, v, g, beta,
                                   o, vh, kh, vh / kh, M, nheads, wait_first);
  };
  cudaError_t e;
  if (ckpt)
    e = M > 1      ? go(gdn_steps_kernel<true, false, 4>, ckpt)
        : wpc == 8 ? go(gdn_steps_kernel<true, true, 8>, ckpt)
                   : go(gdn_steps_kernel<true, true, 4>, ckpt);
  else
    e = M > 1      ? go(gdn_steps_kernel<false, false, 4>, (float *)nullptr)
        : wpc == 8 ? go(gdn_steps_kernel<false, true, 8>, (float *)nullptr)
                   : go(gdn_steps_kernel<false, true, 4>, (float *)nullptr);
  return e;
}

cudaError_t steps_timeouts(unsigned int *count) {
  return cudaMemcpyFromSymbol(count, g_steps_timeouts, sizeof(unsigned int));
}

cudaError_t launch_copy(float *dst, const float *src, size_t n,
                        cudaStream_t stream) {
  const size_t n4 = n / 4;
  if (n4 == 0) return cudaSuccess;
  const size_t blocks = (n4 + 256 * kCopyUnroll - 1) / (256 * kCopyUnroll);
  if (blocks > 0x7fffffffull) return cudaErrorInvalidConfiguration;
  copy_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      reinterpret_cast<float4 *>(dst), reinterpret_cast<const float4 *>(src),
      n4);
  return cudaGetLastError();
}

cudaError_t launch_rollback_seq(float *S, const float *snap, const float *ckpt,
                                const int *m_dev, int *err_dev, int B, int vh,
                                int M, cudaStream_t stream) {
  const size_t nheads = (size_t)B * vh;
  if (nheads == 0) return cudaSuccess;
  if (nheads * kRollTiles > 0x7fffffffull) return cudaErrorInvalidConfiguration;
  rollback_seq_kernel<<<(unsigned)(nheads * kRollTiles), 256, 0, stream>>>(
      reinterpret_cast<float4 *>(S), reinterpret_cast<const float4 *>(snap),
      reinterpret_cast<const float4 *>(ckpt), m_dev, err_dev, vh, M, nheads);
  return cudaGetLastError();
}

}  // namespace gdn
