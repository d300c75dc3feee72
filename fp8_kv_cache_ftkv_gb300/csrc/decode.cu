// decode.cu -- split-K decode attention over the FP8 (E4M3FN) pool, split merge included.
//
// What it computes (FreeToken PR #897, opening description and "Fresh R9700 stage-1 A/B"): for a
// request with n keys and a BF16 query row, per query head i (KV head h = i / G)
//     s_j = (q . k^_j) * sm_scale,   k^_j = decode(codeK_j) * scaleK_j,   v^_j likewise,
//     o   = sum_j softmax(s)_j v^_j,
// with split-K over the keys: each CTA covers one slice of the keys and writes a partial (max, sum,
// accumulator); the last slice of a (request, KV head) to finish merges them in the same launch.
// Multi-row decode: row r of R rows sees keys 0 .. n-R+r.
//
// GB300 design:
//  * CTA = (key slice, KV head, request).  Each warp runs its own software pipeline: cp.async
//    gathers of 16-key blocks (128 B of K codes + 128 B of V codes + two FP32 scales per key) into a
//    private shared-memory ring, so ~150 KB per SM are in flight without CTA-wide barriers.  The slot
//    indices of the slice are staged in shared memory first, so no gather waits on an index load.
//  * QK^T runs on the FP8 tensor cores directly on the stored codes (mma m16n8k32, E4M3 x E4M3 ->
//    FP32): the K codes are the A operand as they sit in memory, no conversion.  The BF16 query is
//    split per head into two E4M3 pieces q = a (h1 + h2/16), a a power of two: h1 is q rounded to 4
//    significant bits and the remainder k * 2^(e-7), |k| <= 8, fits h2 exactly, so every element
//    within 13 binades of the head's largest one is represented without error.  The two partial dot
//    products are recombined in FP32 with the per-key K scale.
//  * PV runs on FP16 tensor cores (m16n8k16): V codes are converted exactly with the packed
//    hardware converter and the V scale is folded into the probabilities, w_j = 2^(s_j - m) * scaleV_j
//    (FP32 products, no logarithms: an added log2(scale) would be rounded to the ulp of a large logit).
//    The softmax maximum is lazy, as in decode_tok.cu: m is raised, and the accumulator rescaled, only
//    when a score exceeds it by more than 8 (a warp vote).  PV accumulates in place: FP16 has a narrow
//    exponent range and the per-row V scales of a slice can span 2^30, so the MMA takes w_j * 2^-E with
//    one power-of-two exponent E per (row, head) that only grows (raised, and the accumulator rescaled
//    exactly, when some w would exceed 2^(E + 12)).  (A normalisation of every 16-key block by its own
//    maximum, with the block's tile added into the accumulator by FMAs, measured 1,241 us against 1,143 us
//    on the batched 64-request launch.)
//  * The 8 query heads of a GQA group are the MMA N dimension, so G = 8 wastes nothing.
#include <cfloat>
#include <mutex>

#include "decode_common.cuh"
#include "decode_merge.cuh"
#include "ftkv_device.cuh"
#include "ftkv_internal.h"

namespace ftkv {
namespace {

constexpr int KB = 16;                       // keys per block (MMA M of QK^T, MMA K of PV)
constexpr int STAGE_K = KB * kHeadDim;       // 2048 B of K codes
constexpr int STAGE_V = KB * kHeadDim;       // 2048 B of V codes
constexpr int STAGE_S = KB * 4 * 2;          // 16 K scales + 16 V scales
constexpr int STAGE_BYTES = STAGE_K + STAGE_V + STAGE_S;
constexpr int MAX_SUB = 4096;                // slot indices staged in shared memory at a time
#ifndef FTKV_MR_TC
#define FTKV_MR_TC 1
#endif
constexpr bool kMultiRowTensorMemory = FTKV_MR_TC != 0;  // multi-row requests: decode_mr.cu
constexpr float kLazyMax = 8.0f;             // log2 slack of the running maximum
constexpr int kLazyExp = 12;                 // w may reach 2^(E + kLazyExp) before E is raised

template <int RPW>
struct Cfg;
template <>
struct Cfg<1> {                               // single-row decode
  static constexpr int WARPS = 16;
  static constexpr int NSTAGE = 3;
};
template <>
struct Cfg<2> {                               // multi-row decode: two query rows per warp
  static constexpr int WARPS = 8;
  static constexpr int NSTAGE = 4;
};

// query pieces of the CTA's rows, shared by all warps: [row][8 heads][2 pieces][128] E4M3 codes, then
// [row][8 heads] FP32 multipliers; rows per request: 1 for RPW = 1, up to 8 (the multi-row cap) for RPW = 2
template <int RPW>
constexpr int q_rows_max() { return RPW == 1 ? 1 : 8; }
template <int RPW>
constexpr int q_area_bytes() { return q_rows_max<RPW>() * 8 * (2 * kHeadDim + 4); }
template <int RPW>
constexpr int smem_bytes() {
  return Cfg<RPW>::WARPS * Cfg<RPW>::NSTAGE * STAGE_BYTES + MAX_SUB * 4 + q_area_bytes<RPW>();
}
static_assert(smem_bytes<1>() <= 227 * 1024, "decode smem");
// in-CTA merge area: per (warp, row, head) 128 accumulators, then per (warp, row, head) m and l, then per
// (row, head) pair the warp weights, M and L; rows per request: 1 for RPW = 1, up to 8 (the multi-row
// cap) for RPW = 2
template <int RPW>
constexpr int merge_area_bytes() {
  return (Cfg<RPW>::WARPS * RPW * 8 * (kHeadDim + 2) + (RPW == 1 ? 1 : 8) * 8 * (Cfg<RPW>::WARPS + 2)) * 4;
}
static_assert(merge_area_bytes<1>() <= Cfg<1>::WARPS * Cfg<1>::NSTAGE * STAGE_BYTES, "merge");
static_assert(merge_area_bytes<2>() <= Cfg<2>::WARPS * Cfg<2>::NSTAGE * STAGE_BYTES, "merge");

// Shared-memory position of 16-byte chunk p of key `key` in a stage.  K rows are read as
// (key g, chunks 2t and 2t+1), V rows as (keys 2t.., chunk g); the XOR swizzles make both reads and
// the cp.async writes bank-conflict free.
__device__ __forceinline__ uint32_t k_chunk_off(int key, int p) { return (key * 8 + (p ^ (key & 1))) * 16; }
__device__ __forceinline__ uint32_t v_chunk_off(int key, int p) { return STAGE_K + (key * 8 + (p ^ (((key >> 1) & 3) << 1))) * 16; }

template <int RPW>
__global__ void __launch_bounds__(Cfg<RPW>::WARPS * 32, 1) decode_split_kernel(const DecodeArgs a) {
  pdl_enter();
  constexpr int WARPS = Cfg<RPW>::WARPS;
  constexpr int NSTAGE = Cfg<RPW>::NSTAGE;
  extern __shared__ __align__(128) uint8_t smem[];
  int32_t* sslot = reinterpret_cast<int32_t*>(smem + WARPS * NSTAGE * STAGE_BYTES);
  uint8_t* qsm = smem + WARPS * NSTAGE * STAGE_BYTES + MAX_SUB * 4;              // query piece codes
  float* qmul = reinterpret_cast<float*>(qsm + q_rows_max<RPW>() * 8 * 2 * kHeadDim);  // their multipliers

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;

  const int64_t n = clamp_seq_len(a, b, threadIdx.x == 0 && split == 0 && h == 0);
  int64_t row0;
  int R;
  if (a.q_row_offsets) {
    row0 = a.q_row_offsets[b];
    R = a.q_row_offsets[b + 1] - a.q_row_offsets[b];
  } else {
    row0 = b;
    R = 1;
  }
  if (R < 0 || R > a.max_q_rows || row0 < 0 || row0 + R > a.total_q_rows) {
    if (threadIdx.x == 0 && split == 0 && h == 0) flag_error(a.err, kDevErrQRows);
    if (a.coop) coop_finish<WARPS>(a);
    return;  // inconsistent row offsets: skip the request rather than read outside q
  }
  if (n == 0) {  // no keys: the rows of this KV head's group are zero
    if (split == 0)
      for (int i = threadIdx.x; i < R * a.group * kHeadDim; i += blockDim.x)
        a.out[((row0 + i / (a.group * kHeadDim)) * a.num_q_heads + h * a.group + (i / kHeadDim) % a.group) *
                  kHeadDim + i % kHeadDim] = 0;
    if (a.coop) coop_finish<WARPS>(a);
    return;
  }
  // key indices fit in 32 bits (the host rejects max_seq_len >= 2^31); slices cover keys [first, n)
  const int kfirst = static_cast<int>(first_key(a, n, R));
  const int j0 = kfirst + split * static_cast<int>(a.chunk);
  const int j1 = (static_cast<int64_t>(j0) + a.chunk < n) ? j0 + static_cast<int>(a.chunk) : static_cast<int>(n);
  if (j0 >= n || R == 0) {  // slices past the end hold no keys and take no ticket
    if (a.coop) coop_finish<WARPS>(a);
    return;
  }

  // ---- warp roles: row group rg (RPW query rows) x key-interleave index kw ----
  const int nrg = (R + RPW - 1) / RPW;
  const int wk = WARPS / nrg;
  const int rg = warp / wk, kw = warp % wk;
  const bool active = rg < nrg;
  int lim[RPW], low[RPW];  // keys low .. lim-1 of this slice are attended by the row
#pragma unroll
  for (int i = 0; i < RPW; i++) {
    const int rabs = rg * RPW + i;
    const bool valid = active && rabs < R;
    const int vis = static_cast<int>(n) - R + rabs + 1;  // keys 0 .. vis-1 are visible to this row
    lim[i] = valid ? (vis < j1 ? vis : j1) : j0;
    low[i] = (a.window > 0 && vis - a.window > 0) ? vis - static_cast<int>(a.window) : 0;  // sliding window
  }

  // The first slot window's indices are requested now and staged after the query pieces, so the two
  // round trips overlap.
  constexpr int PRE = 2;  // slot indices per thread read ahead (1,024 keys per CTA)
  const int nk0 = (j1 - j0 < MAX_SUB) ? j1 - j0 : MAX_SUB;
  int32_t pre[PRE];
#pragma unroll
  for (int u = 0; u < PRE; u++) {
    const int i = threadIdx.x + u * blockDim.x;
    pre[u] = (i < nk0) ? a.req_to_slot[static_cast<int64_t>(b) * a.req_stride + j0 + i] : 0;
  }

  // ---- fused store: the request's new tokens (positions n-R .. n-1) that fall in this slice are
  // quantized into the pool first, one warp per token (K row on lanes 0-15, V row on 16-31) with the
  // store kernel's arithmetic, starting from the upper half of the warps while the lower half computes
  // the query pieces.  The barrier after the pieces orders these writes before every warp's loads, which
  // then read the new rows like any other key. ----
  if (a.k_new) {
    const int nq0 = static_cast<int>(n) - R;  // position of the request's first new token
    const int first = (nq0 > j0) ? nq0 : j0;
    if (first < j1) {  // CTA-uniform
      bool wrote = false;
      for (int pos = ((first > 0) ? first : 0) + (warp + WARPS / 2) % WARPS; pos < j1; pos += WARPS) {  // warp-uniform
        const int half = lane >> 4, l = lane & 15;
        const uint16_t* src =
            (half ? a.v_new : a.k_new) + ((row0 + pos - nq0) * a.num_kv_heads + h) * kHeadDim + l * 8;
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src));
        const int32_t sv = a.req_to_slot[static_cast<int64_t>(b) * a.req_stride + pos];
        float sc;
        const uint2 packed = quantize_row_lane8(raw, sc);
        if (sv >= 0 && sv < a.num_rows) {  // a bad slot is flagged when staged; nothing is written
          const int64_t row = static_cast<int64_t>(sv) * a.num_kv_heads + h;
          // the pool is the caller's writable memory (ftkv_pool holds non-const pointers)
          *reinterpret_cast<uint2*>(const_cast<uint8_t*>(half ? a.v_codes : a.k_codes) + row * kHeadDim + l * 8) =
              packed;
          if (l == 0) const_cast<float*>(half ? a.v_scales : a.k_scales)[row] = sc;
        }
        wrote = true;
      }
      if (wrote) __threadfence();  // the rows reach L2 before the barrier below
    }
  }

  // ---- query pieces, computed once per CTA: one warp per (row, head), 4 d values per lane ----
  // x = q * 2^(7-ex), ex the exponent of max|q| over the head, has |x| < 256; pieces x = h1 + h2/16, both
  // E4M3 (exact unless |q| < 2^-13 max|q|); multiplier 2^(ex-7) * sm_scale * log2(e).  Heads past the group
  // (padding of the 8-wide MMA N dimension) get zero pieces.
  for (int pr = warp; pr < R * 8; pr += WARPS) {  // warp-uniform
    const int rr = pr >> 3, hq = pr & 7;
    float x[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (hq < a.group) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(
          a.q + ((row0 + rr) * a.num_q_heads + h * a.group + hq) * kHeadDim + 4 * lane));
      x[0] = bf16_lo(v.x);
      x[1] = bf16_hi(v.x);
      x[2] = bf16_lo(v.y);
      x[3] = bf16_hi(v.y);
    }
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    int ex = (amax > 0.0f) ? ilogbf(amax) : 0;
    ex = ex < -120 ? -120 : ex;
    const float up = __uint_as_float(static_cast<uint32_t>(127 + 7 - ex) << 23);
#pragma unroll
    for (int e = 0; e < 4; e++) x[e] *= up;
    uint8_t* dst = qsm + (rr * 8 + hq) * 2 * kHeadDim + 4 * lane;
#pragma unroll
    for (int p = 0; p < 2; p++) {
      const uint32_t c01 = e4m3x2_encode(x[0], x[1]), c23 = e4m3x2_encode(x[2], x[3]);
      *reinterpret_cast<uint32_t*>(dst + p * kHeadDim) = c01 | (c23 << 16);
      if (p == 0) {
        const float2 v01 = f16x2_to_float2(e4m3x2_to_f16x2(c01));
        const float2 v23 = f16x2_to_float2(e4m3x2_to_f16x2(c23));
        x[0] = (x[0] - v01.x) * 16.0f;
        x[1] = (x[1] - v01.y) * 16.0f;
        x[2] = (x[2] - v23.x) * 16.0f;
        x[3] = (x[3] - v23.y) * 16.0f;
      }
    }
    if (lane == 0) qmul[rr * 8 + hq] = __uint_as_float(static_cast<uint32_t>(127 - 7 + ex) << 23) * a.qk_scale_log2;
  }
  __syncthreads();
  // B operand of QK^T for this warp's rows: head g, d = 32t + 8kk + {0..3} (b0) / {4..7} (b1)
  uint32_t qp[RPW][2][4][2];
  float fq[RPW][2];  // per-head multiplier for heads 2t, 2t+1
#pragma unroll
  for (int i = 0; i < RPW; i++) {
    const int rabs = rg * RPW + i;
    const bool valid = active && rabs < R;
    const int rsafe = valid ? rabs : 0;
    const uint32_t src = smem_addr(qsm) + (rsafe * 8 + g) * 2 * kHeadDim + 32 * t;
#pragma unroll
    for (int p = 0; p < 2; p++) {
      const uint4 w0 = valid ? ld_shared_v4(src + p * kHeadDim) : make_uint4(0, 0, 0, 0);
      const uint4 w1 = valid ? ld_shared_v4(src + p * kHeadDim + 16) : make_uint4(0, 0, 0, 0);
      qp[i][p][0][0] = w0.x; qp[i][p][0][1] = w0.y; qp[i][p][1][0] = w0.z; qp[i][p][1][1] = w0.w;
      qp[i][p][2][0] = w1.x; qp[i][p][2][1] = w1.y; qp[i][p][3][0] = w1.z; qp[i][p][3][1] = w1.w;
    }
    fq[i][0] = valid ? qmul[rsafe * 8 + 2 * t] : 0.0f;
    fq[i][1] = valid ? qmul[rsafe * 8 + 2 * t + 1] : 0.0f;
  }

  float acc[RPW][8][4];         // in units of 2^E
  float m[RPW][2], l[RPW][2];   // running (lazy) max of s (log2 units) and running sum of 2^(s - m)
  int E[RPW][2];                // FP16 operand exponent: PV takes w * 2^-E
  float wlim[RPW][2], iw[RPW][2];
#pragma unroll
  for (int i = 0; i < RPW; i++) {
#pragma unroll
    for (int mt = 0; mt < 8; mt++) acc[i][mt][0] = acc[i][mt][1] = acc[i][mt][2] = acc[i][mt][3] = 0.0f;
#pragma unroll
    for (int hx = 0; hx < 2; hx++) {
      m[i][hx] = -INFINITY;
      l[i][hx] = 0.0f;
      E[i][hx] = -126;
      wlim[i][hx] = exp2i(-126 + kLazyExp);
      iw[i][hx] = exp2i(126);
    }
  }

  const uint32_t ring = smem_addr(smem) + warp * NSTAGE * STAGE_BYTES;
  const int64_t hkv = a.num_kv_heads;

  for (int js = j0; js < j1; js += MAX_SUB) {
    const int je = (js + MAX_SUB < j1) ? js + MAX_SUB : j1;
    const int nk = je - js;
    __syncthreads();  // every warp is done with the previous slot window
    auto stage_slot = [&](int i, int32_t sv) {
      if (sv < 0 || sv >= a.num_rows) {
        flag_error(a.err, kDevErrBadSlot);
        sv = 0;
      }
      sslot[i] = sv;
    };
    int i = threadIdx.x;
    if (js == j0) {  // the indices read ahead: i < nk0 == nk
#pragma unroll
      for (int u = 0; u < PRE; u++, i += blockDim.x)
        if (i < nk) stage_slot(i, pre[u]);
    }
    for (; i < nk; i += blockDim.x) stage_slot(i, a.req_to_slot[static_cast<int64_t>(b) * a.req_stride + js + i]);
    __syncthreads();
    if (!active) continue;

    const int nblk = (nk + KB - 1) / KB;
    const int my_nblk = nblk > kw ? (nblk - kw + wk - 1) / wk : 0;

    auto issue = [&](int i) {
      if (i < my_nblk) {
        const int key0 = (kw + i * wk) * KB;
        const uint32_t st = ring + (i % NSTAGE) * STAGE_BYTES;
        const int p = lane & 7;
#pragma unroll
        for (int r = 0; r < 4; r++) {
          const int key = (lane >> 3) + 4 * r;
          if (key0 + key < nk) {
            const int64_t off = (static_cast<int64_t>(sslot[key0 + key]) * hkv + h) * kHeadDim + p * 16;
            cp_async_16(st + k_chunk_off(key, p), a.k_codes + off);
            cp_async_16(st + v_chunk_off(key, p), a.v_codes + off);
          } else {
            st_shared_zero16(st + k_chunk_off(key, p));
            st_shared_zero16(st + v_chunk_off(key, p));
          }
        }
        const int key = lane & 15;
        const uint32_t ds = st + STAGE_K + STAGE_V + lane * 4;
        if (key0 + key < nk) {
          const int64_t row = static_cast<int64_t>(sslot[key0 + key]) * hkv + h;
          cp_async_4(ds, (lane < 16 ? a.k_scales : a.v_scales) + row);
        } else {
          st_shared_u32(ds, 0u);
        }
      }
      cp_async_commit();
    };

#pragma unroll 1
    for (int i = 0; i < NSTAGE - 1; i++) issue(i);

#pragma unroll 1
    for (int i = 0; i < my_nblk; i++) {
      issue(i + NSTAGE - 1);
      cp_async_wait<NSTAGE - 1>();
      __syncwarp();
      const uint32_t st = ring + (i % NSTAGE) * STAGE_BYTES;
      const int jb = js + (kw + i * wk) * KB;

      // ---- S^T = K Q^T on E4M3 codes: keys as M (rows g, g+8), heads as N, 2 query pieces ----
      const uint4 kA0 = ld_shared_v4(st + k_chunk_off(g, 2 * t));
      const uint4 kA1 = ld_shared_v4(st + k_chunk_off(g, 2 * t + 1));
      const uint4 kB0 = ld_shared_v4(st + k_chunk_off(g + 8, 2 * t));
      const uint4 kB1 = ld_shared_v4(st + k_chunk_off(g + 8, 2 * t + 1));
      float c[RPW][2][4];
#pragma unroll
      for (int r = 0; r < RPW; r++)
#pragma unroll
        for (int p = 0; p < 2; p++) c[r][p][0] = c[r][p][1] = c[r][p][2] = c[r][p][3] = 0.0f;
#pragma unroll
      for (int kk = 0; kk < 4; kk++) {
        const uint4& A = kk < 2 ? kA0 : kA1;
        const uint4& B = kk < 2 ? kB0 : kB1;
        const uint32_t a0 = word(A, 2 * (kk & 1)), a2 = word(A, 2 * (kk & 1) + 1);
        const uint32_t a1 = word(B, 2 * (kk & 1)), a3 = word(B, 2 * (kk & 1) + 1);
#pragma unroll
        for (int r = 0; r < RPW; r++)
#pragma unroll
          for (int p = 0; p < 2; p++) mma_e4m3_16832(c[r][p], a0, a1, a2, a3, qp[r][p][kk][0], qp[r][p][kk][1]);
      }

      // ---- per-key scales ----
      const uint32_t ss = st + STAGE_K + STAGE_V;
      const float skg = ld_shared_f32(ss + g * 4), skg8 = ld_shared_f32(ss + (g + 8) * 4);
      const float svg = ld_shared_f32(ss + 64 + g * 4), svg8 = ld_shared_f32(ss + 64 + (g + 8) * 4);

      // ---- softmax with a lazy maximum (log2 domain): m is raised, and the accumulator rescaled, only when a score
      // exceeds it by more than kLazyMax (a warp vote); P' = p * scaleV * 2^-E into the B fragments of PV, with
      // one power-of-two exponent E per (row, head) that only grows (raised, and the accumulator rescaled exactly,
      // when some w would exceed 2^(E + kLazyExp)) ----
      const int jg = jb + g, jg8 = jb + g + 8;
      uint32_t pb0[RPW], pb1[RPW];
#pragma unroll
      for (int r = 0; r < RPW; r++) {
        const int lr = lim[r] < je ? lim[r] : je;
        float dot[4];
#pragma unroll
        for (int e = 0; e < 4; e++) dot[e] = fmaf(c[r][1][e], 1.0f / 16.0f, c[r][0][e]);
        const bool in0 = jg < lr && jg >= low[r], in8 = jg8 < lr && jg8 >= low[r];
        const float s0 = in0 ? dot[0] * (skg * fq[r][0]) : -INFINITY;
        const float s1 = in0 ? dot[1] * (skg * fq[r][1]) : -INFINITY;
        const float s2 = in8 ? dot[2] * (skg8 * fq[r][0]) : -INFINITY;
        const float s3 = in8 ? dot[3] * (skg8 * fq[r][1]) : -INFINITY;
        const bool raise = fmaxf(s0, s2) > m[r][0] + kLazyMax || fmaxf(s1, s3) > m[r][1] + kLazyMax;
        if (__any_sync(0xffffffffu, raise)) {  // new maximum: exact block max, rescale
          float bm0 = fmaxf(s0, s2), bm1 = fmaxf(s1, s3);
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
            bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
          }
          const float mn0 = fmaxf(m[r][0], bm0), mn1 = fmaxf(m[r][1], bm1);
          const float al0 = (m[r][0] == -INFINITY) ? 1.0f : fast_exp2(m[r][0] - mn0);
          const float al1 = (m[r][1] == -INFINITY) ? 1.0f : fast_exp2(m[r][1] - mn1);
          m[r][0] = mn0;
          m[r][1] = mn1;
          l[r][0] *= al0;
          l[r][1] *= al1;
#pragma unroll
          for (int mt = 0; mt < 8; mt++) {
            acc[r][mt][0] *= al0;
            acc[r][mt][1] *= al1;
            acc[r][mt][2] *= al0;
            acc[r][mt][3] *= al1;
          }
        }
        const float mu0 = (m[r][0] == -INFINITY) ? 0.0f : m[r][0], mu1 = (m[r][1] == -INFINITY) ? 0.0f : m[r][1];
        const float p0 = fast_exp2(s0 - mu0), p1 = fast_exp2(s1 - mu1);
        const float p2 = fast_exp2(s2 - mu0), p3 = fast_exp2(s3 - mu1);
        l[r][0] += p0 + p2;
        l[r][1] += p1 + p3;
        const float w0 = p0 * svg, w1 = p1 * svg, w2 = p2 * svg8, w3 = p3 * svg8;
        const bool grow = fmaxf(w0, w2) > wlim[r][0] || fmaxf(w1, w3) > wlim[r][1];
        if (__any_sync(0xffffffffu, grow)) {
          float W0 = fmaxf(w0, w2), W1 = fmaxf(w1, w3);
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            W0 = fmaxf(W0, __shfl_xor_sync(0xffffffffu, W0, off));
            W1 = fmaxf(W1, __shfl_xor_sync(0xffffffffu, W1, off));
          }
          // exponent of W (a subnormal W counts as -126); E never decreases
          const int e0 = max(E[r][0], max(static_cast<int>(__float_as_uint(W0) >> 23), 1) - 127);
          const int e1 = max(E[r][1], max(static_cast<int>(__float_as_uint(W1) >> 23), 1) - 127);
          const int ne0 = min(e0, 127 - kLazyExp), ne1 = min(e1, 127 - kLazyExp);
          // <= 1, exact (0 below 2^-126: the earlier terms vanish next to the new ones)
          const float f0 = (E[r][0] - ne0 < -126) ? 0.0f : exp2i(E[r][0] - ne0);
          const float f1 = (E[r][1] - ne1 < -126) ? 0.0f : exp2i(E[r][1] - ne1);
          E[r][0] = ne0;
          E[r][1] = ne1;
          wlim[r][0] = exp2i(ne0 + kLazyExp);
          wlim[r][1] = exp2i(ne1 + kLazyExp);
          iw[r][0] = exp2i(-ne0);
          iw[r][1] = exp2i(-ne1);
#pragma unroll
          for (int mt = 0; mt < 8; mt++) {
            acc[r][mt][0] *= f0;
            acc[r][mt][1] *= f1;
            acc[r][mt][2] *= f0;
            acc[r][mt][3] *= f1;
          }
        }
        pb0[r] = movmatrix_trans(float2_to_f16x2(w0 * iw[r][0], w1 * iw[r][1]));   // keys 0..7
        pb1[r] = movmatrix_trans(float2_to_f16x2(w2 * iw[r][0], w3 * iw[r][1]));   // keys 8..15
      }

      // ---- O^T += V^T P'^T : d as M (d = 16g + 2mt [+1]), heads as N, keys as K ----
      const uint4 v0 = ld_shared_v4(st + v_chunk_off(2 * t, g));
      const uint4 v1 = ld_shared_v4(st + v_chunk_off(2 * t + 1, g));
      const uint4 v8 = ld_shared_v4(st + v_chunk_off(2 * t + 8, g));
      const uint4 v9 = ld_shared_v4(st + v_chunk_off(2 * t + 9, g));
#pragma unroll
      for (int w = 0; w < 4; w++) {
        const uint32_t x0 = word(v0, w), x1 = word(v1, w), x8 = word(v8, w), x9 = word(v9, w);
        const uint32_t lo01 = prmt(x0, x1, 0x5140), hi01 = prmt(x0, x1, 0x7362);
        const uint32_t lo89 = prmt(x8, x9, 0x5140), hi89 = prmt(x8, x9, 0x7362);
        {
          const uint32_t a0 = e4m3_lo2(lo01), a1 = e4m3_hi2(lo01);
          const uint32_t a2 = e4m3_lo2(lo89), a3 = e4m3_hi2(lo89);
#pragma unroll
          for (int r = 0; r < RPW; r++) mma_f16_16816(acc[r][2 * w], a0, a1, a2, a3, pb0[r], pb1[r]);
        }
        {
          const uint32_t a0 = e4m3_lo2(hi01), a1 = e4m3_hi2(hi01);
          const uint32_t a2 = e4m3_lo2(hi89), a3 = e4m3_hi2(hi89);
#pragma unroll
          for (int r = 0; r < RPW; r++) mma_f16_16816(acc[r][2 * w + 1], a0, a1, a2, a3, pb0[r], pb1[r]);
        }
      }
      __syncwarp();
    }
    cp_async_wait<0>();
  }

  // ---- finalize this warp: full row sums; the accumulator brought from units of 2^E to units of 2^m ----
#pragma unroll
  for (int r = 0; r < RPW; r++)
#pragma unroll
    for (int hh = 0; hh < 2; hh++) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) l[r][hh] += __shfl_xor_sync(0xffffffffu, l[r][hh], off);
      const float up = exp2i(E[r][hh]);
#pragma unroll
      for (int mt = 0; mt < 8; mt++) {
        acc[r][mt][hh] *= up;
        acc[r][mt][2 + hh] *= up;
      }
    }

  __syncthreads();  // the rings are free: reuse them as the merge area
  // ---- merge the wk warps of each row group into this slice's partial ----
  // Accumulator rows hold 32 float4 chunks; chunk c of head hd sits at c ^ ((hd >> 1) & 3), which makes
  // the stores (lanes g, t write chunk 4g + q of heads 2t, 2t+1) and the loads of the sums (consecutive
  // chunks of one head) free of bank conflicts.
  float* macc = reinterpret_cast<float*>(smem);              // [warp][row][head][128]
  float* wml = macc + WARPS * RPW * 8 * kHeadDim;             // [warp][row][head][2]: m, l
  float* mw = wml + WARPS * RPW * 8 * 2;                      // per (row, head) pair: wk weights, then M, L
  if (active) {
#pragma unroll
    for (int r = 0; r < RPW; r++) {
#pragma unroll
      for (int hh = 0; hh < 2; hh++) {
        const int hd = 2 * t + hh;
        float4* dst = reinterpret_cast<float4*>(macc + ((warp * RPW + r) * 8 + hd) * kHeadDim);
        // head hd: d = 16g + 2mt -> acc[mt][hh], d = 16g + 2mt + 1 -> acc[mt][2+hh]; chunk 4g + q4 holds
        // d = 16g + 4q4 .. 16g + 4q4 + 3
#pragma unroll
        for (int q4 = 0; q4 < 4; q4++)
          dst[(4 * g + q4) ^ t] = make_float4(acc[r][2 * q4][hh], acc[r][2 * q4][2 + hh], acc[r][2 * q4 + 1][hh],
                                               acc[r][2 * q4 + 1][2 + hh]);
        if (g == 0) {
          wml[((warp * RPW + r) * 8 + hd) * 2] = m[r][hh];
          wml[((warp * RPW + r) * 8 + hd) * 2 + 1] = l[r][hh];
        }
      }
    }
  }
  __syncthreads();
  // weights: one warp per (row, head) pair, lane k holding warp k's maximum and sum; M and L by warp
  // reductions, weights 2^(m_k - M)
  const int npairs = R * a.group;
  constexpr int WSTRIDE = WARPS + 2;
  for (int pr = warp; pr < npairs; pr += WARPS) {
    const int rr = pr / a.group, hh = pr % a.group;
    const int rgi = rr / RPW, r = rr % RPW;
    const bool has = lane < wk;
    const int idx = has ? (((rgi * wk + lane) * RPW + r) * 8 + hh) * 2 : 0;
    const float mk = has ? wml[idx] : -INFINITY;
    float M = mk;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float wt = (has && M != -INFINITY) ? exp2f(mk - M) : 0.0f;
    float L = has ? wt * wml[idx + 1] : 0.0f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    float* w = mw + pr * WSTRIDE;
    if (has) w[lane] = wt;
    if (lane == 0) {
      w[WARPS] = M;
      w[WARPS + 1] = L;
    }
  }
  __syncthreads();
  // sums: item (pair, chunk) split over two adjacent lanes, even and odd warps, joined by one shuffle;
  // npairs * 64 and blockDim.x are multiples of 32, so a warp is either fully inside the range or outside
  constexpr int KSTEP4 = RPW * 8 * kHeadDim / 4;  // float4s from warp k to warp k + 1 of the row group
  for (int it = threadIdx.x; it < npairs * 64; it += blockDim.x) {
    const int half = it & 1, c = (it >> 1) & 31, pr = it >> 6;
    const int rr = pr / a.group, hh = pr - rr * a.group;
    const int rgi = rr / RPW, r = rr - rgi * RPW;
    const float* w = mw + pr * WSTRIDE;
    const float4* src = reinterpret_cast<const float4*>(macc + ((rgi * wk * RPW + r) * 8 + hh) * kHeadDim) +
                        (c ^ ((hh >> 1) & 3));
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < WARPS; k += 2) {
      if (k + half < wk) {
        const float4 v = src[(k + half) * KSTEP4];
        const float wv = w[k + half];
        A.x = fmaf(wv, v.x, A.x);
        A.y = fmaf(wv, v.y, A.y);
        A.z = fmaf(wv, v.z, A.z);
        A.w = fmaf(wv, v.w, A.w);
      }
    }
    A.x += __shfl_xor_sync(0xffffffffu, A.x, 1);
    A.y += __shfl_xor_sync(0xffffffffu, A.y, 1);
    A.z += __shfl_xor_sync(0xffffffffu, A.z, 1);
    A.w += __shfl_xor_sync(0xffffffffu, A.w, 1);
    if (half == 0) {
      const int64_t prow = ((row0 + rr) * a.num_q_heads + h * a.group + hh) * a.num_splits * a.pps + split;
      reinterpret_cast<float4*>(a.part_acc + prow * kHeadDim)[c] = A;
      if (c == 0) {
        a.part_ml[prow * 2] = w[WARPS];
        a.part_ml[prow * 2 + 1] = w[WARPS + 1];
      }
    }
  }

  if (a.coop) {
    coop_finish<WARPS>(a);
    return;
  }
  // ---- split merge, done by the last slice of (request, KV head) to arrive ----
  // Every slice publishes its partial, then takes a ticket; the CTA that draws the last ticket merges
  // all slices (o = sum_s 2^(M_s - M) A_s / sum_s 2^(M_s - M) L_s) and resets the counter for the
  // next call.  Nothing ever waits on another CTA.
  __shared__ int s_last;
  const int64_t nsl64 = (n - kfirst + a.chunk - 1) / a.chunk;
  const int nslices = static_cast<int>(nsl64 < a.num_splits ? nsl64 : a.num_splits);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int* ctr = a.counters + static_cast<int64_t>(b) * a.num_kv_heads + h;
    const int prev = atomicAdd(ctr, 1);
    s_last = (prev == nslices - 1);
    if (s_last) *ctr = 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  merge_split_partials(a, row0, R, h, nslices, smem, WARPS * NSTAGE * STAGE_BYTES);  // the ring is idle now
}

template <int RPW>
cudaError_t launch_split(const DecodeArgs& a, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDecodeDevices) return cudaErrorInvalidDevice;
  // per-device set-up, once: dynamic shared memory above 48 KB and the co-resident CTA count (0: no
  // cooperative launch); a grid that fits on the GPU at once is launched cooperatively and merges after a
  // grid barrier
  static std::once_flag once[kMaxDecodeDevices];
  static cudaError_t setup_err[kMaxDecodeDevices];
  static int resident[kMaxDecodeDevices];
  std::call_once(once[dev], [&] {
    setup_err[dev] = cudaFuncSetAttribute(decode_split_kernel<RPW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          smem_bytes<RPW>());
    int coop_ok = 0, sms = 0, per_sm = 0;
    if (setup_err[dev] == cudaSuccess) setup_err[dev] = cudaDeviceGetAttribute(&coop_ok, cudaDevAttrCooperativeLaunch, dev);
    if (setup_err[dev] == cudaSuccess) setup_err[dev] = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (setup_err[dev] == cudaSuccess &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_split_kernel<RPW>, Cfg<RPW>::WARPS * 32,
                                                      smem_bytes<RPW>()) != cudaSuccess)
      per_sm = 0;
    resident[dev] = (coop_ok && per_sm > 0 && sms > 0) ? per_sm * sms : 0;
  });
  if (setup_err[dev] != cudaSuccess) return setup_err[dev];
  dim3 grid(a.num_splits, a.num_kv_heads, a.batch);
  DecodeArgs c = a;
  c.pps = 1;  // one partial per key slice
  const int64_t ctas = int64_t(grid.x) * grid.y * grid.z;
  c.coop = (resident[dev] > 0 && ctas <= resident[dev]) ? 1 : 0;
  if (c.coop) return launch_k_coop(decode_split_kernel<RPW>, grid, dim3(Cfg<RPW>::WARPS * 32), smem_bytes<RPW>(), s, c);
  return launch_k(decode_split_kernel<RPW>, grid, dim3(Cfg<RPW>::WARPS * 32), smem_bytes<RPW>(), s, c);
}

}  // namespace

int decode_ctas_per_sm(int max_q_rows) {
  // the token-major single-row kernel fits two CTAs per SM; the multi-row kernel is shared-memory bound at one
  return max_q_rows <= 1 ? 2 : 1;
}

// Single-row batches: the token-major kernel (decode_tok.cu); multi-row batches: this kernel.
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  if (a.max_q_rows <= 1) return launch_decode_tok(a, s);
  if (kMultiRowTensorMemory) return launch_decode_mr(a, s);
  return launch_split<2>(a, s);
}

}  // namespace ftkv
