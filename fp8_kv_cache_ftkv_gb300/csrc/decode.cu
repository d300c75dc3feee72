// decode.cu -- split-K decode attention over the FP8 (E4M3FN) pool, plus the split merge.
//
// What it computes (FreeToken PR #897, opening description and "Fresh R9700 stage-1 A/B"): for a
// request with n keys and a BF16 query row, per query head i (KV head h = i / G)
//     s_j = (q . k^_j) * sm_scale,   k^_j = decode(codeK_j) * scaleK_j,   v^_j likewise,
//     o   = sum_j softmax(s)_j v^_j,
// with split-K over the keys: a stage-1 kernel covers one slice of the keys per CTA and writes a
// partial (max, sum, accumulator); a merge kernel combines the slices.  Multi-row decode: row r of
// R rows sees keys 0 .. n-R+r.
//
// GB300 design:
//  * CTA = (key slice, KV head, request).  Each warp runs its own software pipeline: cp.async
//    gathers of 16-key blocks (128 B of K codes + 128 B of V codes + two FP32 scales per key) into a
//    private 3-4 stage shared-memory ring, so 100+ KB per SM are in flight with no CTA barriers.
//  * The slot indices of the CTA's slice are staged in shared memory first, so the gathers never
//    wait on a dependent index load.
//  * QK^T and PV are warp-level tensor-core MMAs (m16n8k16, FP16 inputs, FP32 accumulation).  The 8
//    query heads of a GQA group are the MMA's N dimension, so no padding is wasted at G = 8.
//    E4M3 codes become FP16 exactly with the packed hardware converter; the per-key scales are applied
//    to the FP32 scores (K) and folded into the probabilities (V) instead of the codes.
//  * V scales vary over many binades; P*scaleV is kept in FP16 range by tracking the running maximum
//    binary exponent E of the V scales of a slice (P' = p * scaleV * 2^-E <= 2) and rescaling the
//    accumulator when E grows -- an exact power-of-two bookkeeping next to the usual running max.
//  * Queries are scaled by a power of two per head so the FP16 copy of a BF16 query is exact.
#include <cfloat>

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
constexpr int MERGE_STRIDE = 132;            // floats per (warp, row, head) in the merge area

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

template <int RPW>
constexpr int smem_bytes() {
  return Cfg<RPW>::WARPS * Cfg<RPW>::NSTAGE * STAGE_BYTES + MAX_SUB * 4;
}
static_assert(smem_bytes<1>() <= 227 * 1024, "decode smem");
static_assert(Cfg<1>::WARPS * 1 * 8 * MERGE_STRIDE * 4 <= Cfg<1>::WARPS * Cfg<1>::NSTAGE * STAGE_BYTES, "merge");
static_assert(Cfg<2>::WARPS * 2 * 8 * MERGE_STRIDE * 4 <= Cfg<2>::WARPS * Cfg<2>::NSTAGE * STAGE_BYTES, "merge");

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Shared-memory position of 16-byte chunk p of key `key` in a stage (XOR swizzles chosen so the
// fragment reads below are conflict-free: K rows are read by (key g, chunk t), V rows by (key 2t.., chunk g)).
__device__ __forceinline__ uint32_t k_chunk_off(int key, int p) { return (key * 8 + (p ^ ((key & 1) << 2))) * 16; }
__device__ __forceinline__ uint32_t v_chunk_off(int key, int p) { return STAGE_K + (key * 8 + (p ^ (((key >> 1) & 3) << 1))) * 16; }

__device__ __forceinline__ int64_t clamp_seq_len(const DecodeArgs& a, int b, bool report) {
  int64_t n = a.seq_lens[b];
  const int64_t nmax = a.max_seq_len < a.req_stride ? a.max_seq_len : a.req_stride;
  if (n < 0 || n > nmax) {
    if (report) flag_error(a.err, kDevErrSeqLen);
    n = n < 0 ? 0 : nmax;
  }
  return n;
}

template <int RPW>
__global__ void __launch_bounds__(Cfg<RPW>::WARPS * 32, 1) decode_split_kernel(const DecodeArgs a) {
  constexpr int WARPS = Cfg<RPW>::WARPS;
  constexpr int NSTAGE = Cfg<RPW>::NSTAGE;
  extern __shared__ __align__(128) uint8_t smem[];
  int32_t* sslot = reinterpret_cast<int32_t*>(smem + WARPS * NSTAGE * STAGE_BYTES);

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
    return;  // inconsistent row offsets: skip the request rather than read outside q
  }
  const int64_t j0 = static_cast<int64_t>(split) * a.chunk;
  const int64_t j1 = (j0 + a.chunk < n) ? j0 + a.chunk : n;
  if (j0 >= n || R == 0) return;  // the merge only reads slices that hold keys

  // ---- warp roles: row group rg (RPW query rows) x key-interleave index kw ----
  const int nrg = (R + RPW - 1) / RPW;
  const int wk = WARPS / nrg;
  const int rg = warp / wk, kw = warp % wk;
  const bool active = rg < nrg;
  int rabs[RPW];
  bool rvalid[RPW];
  int64_t lim[RPW];
#pragma unroll
  for (int i = 0; i < RPW; i++) {
    rabs[i] = rg * RPW + i;
    rvalid[i] = active && rabs[i] < R;
    const int64_t vis = n - R + rabs[i] + 1;  // keys 0 .. vis-1 are visible to this row
    lim[i] = rvalid[i] ? (vis < j1 ? vis : j1) : j0;
  }

  // ---- query fragments (B operand of QK^T): head g of the group, d = 64c + 16t + 4sub + {0..3} ----
  uint32_t qf[RPW][8][2];
  float fq[RPW][2];  // per-head score multiplier for heads 2t, 2t+1: 2^Eq * sm_scale * log2(e)
#pragma unroll
  for (int i = 0; i < RPW; i++) {
    float qv[32];
    float amax = 0.0f;
    if (rvalid[i] && g < a.group) {
      const uint16_t* qp = a.q + ((row0 + rabs[i]) * a.num_q_heads + h * a.group + g) * kHeadDim;
      const uint4 q0 = __ldg(reinterpret_cast<const uint4*>(qp + 16 * t));
      const uint4 q1 = __ldg(reinterpret_cast<const uint4*>(qp + 16 * t + 8));
      const uint4 q2 = __ldg(reinterpret_cast<const uint4*>(qp + 64 + 16 * t));
      const uint4 q3 = __ldg(reinterpret_cast<const uint4*>(qp + 64 + 16 * t + 8));
      const uint4 qq[4] = {q0, q1, q2, q3};
#pragma unroll
      for (int u = 0; u < 4; u++)
#pragma unroll
        for (int w = 0; w < 4; w++) {
          qv[u * 8 + 2 * w] = bf16_lo(word(qq[u], w));
          qv[u * 8 + 2 * w + 1] = bf16_hi(word(qq[u], w));
        }
#pragma unroll
      for (int e = 0; e < 32; e++) amax = fmaxf(amax, fabsf(qv[e]));
    } else {
#pragma unroll
      for (int e = 0; e < 32; e++) qv[e] = 0.0f;
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    int ex = (amax > 0.0f) ? ilogbf(amax) : 0;
    ex = ex < -112 ? -112 : ex;
    const float up = __uint_as_float(static_cast<uint32_t>(127 + 14 - ex) << 23);       // 2^(14-ex)
    const float down = __uint_as_float(static_cast<uint32_t>(127 - 14 + ex) << 23) * a.qk_scale_log2;
    // qv[e]: e in [0,16) -> d = 16t + e ; e in [16,32) -> d = 64 + 16t + (e-16)
#pragma unroll
    for (int c = 0; c < 2; c++)
#pragma unroll
      for (int sub = 0; sub < 4; sub++) {
        const int e = c * 16 + 4 * sub;
        qf[i][4 * c + sub][0] = float2_to_f16x2(qv[e] * up, qv[e + 1] * up);
        qf[i][4 * c + sub][1] = float2_to_f16x2(qv[e + 2] * up, qv[e + 3] * up);
      }
    fq[i][0] = __shfl_sync(0xffffffffu, down, (2 * t) * 4);
    fq[i][1] = __shfl_sync(0xffffffffu, down, (2 * t + 1) * 4);
  }

  float acc[RPW][8][4];
  float m[RPW][2], l[RPW][2];
#pragma unroll
  for (int i = 0; i < RPW; i++) {
#pragma unroll
    for (int mt = 0; mt < 8; mt++) acc[i][mt][0] = acc[i][mt][1] = acc[i][mt][2] = acc[i][mt][3] = 0.0f;
    m[i][0] = m[i][1] = -INFINITY;
    l[i][0] = l[i][1] = 0.0f;
  }
  int bexp = 0;  // running max of the biased FP32 exponent of the V scales seen by this warp

  const uint32_t ring = smem_addr(smem) + warp * NSTAGE * STAGE_BYTES;
  const int64_t hkv = a.num_kv_heads;

  for (int64_t js = j0; js < j1; js += MAX_SUB) {
    const int64_t je = (js + MAX_SUB < j1) ? js + MAX_SUB : j1;
    const int nk = static_cast<int>(je - js);
    __syncthreads();  // every warp is done with the previous slot window
    for (int i = threadIdx.x; i < nk; i += blockDim.x) {
      int32_t s = a.req_to_slot[static_cast<int64_t>(b) * a.req_stride + js + i];
      if (s < 0 || s >= a.num_rows) {
        flag_error(a.err, kDevErrBadSlot);
        s = 0;
      }
      sslot[i] = s;
    }
    __syncthreads();
    if (!active) continue;

    const int nblk = (nk + KB - 1) / KB;
    const int my_nblk = nblk > kw ? (nblk - kw + wk - 1) / wk : 0;

    auto issue = [&](int i) {
      if (i < my_nblk) {
        const int key0 = (kw + i * wk) * KB;
        const uint32_t st = ring + (i % NSTAGE) * STAGE_BYTES;
#pragma unroll
        for (int r = 0; r < 4; r++) {
          const int key = (lane >> 3) + 4 * r;
          const int p = lane & 7;
          if (key0 + key < nk) {
            const int64_t row = static_cast<int64_t>(sslot[key0 + key]) * hkv + h;
            cp_async_16(st + k_chunk_off(key, p), a.k_codes + row * kHeadDim + p * 16);
            cp_async_16(st + v_chunk_off(key, p), a.v_codes + row * kHeadDim + p * 16);
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
      const int64_t jb = js + static_cast<int64_t>(kw + i * wk) * KB;

      // ---- S^T = K Q^T : keys as M (rows g, g+8), query heads as N ----
      const uint4 kA0 = ld_shared_v4(st + k_chunk_off(g, t));
      const uint4 kA1 = ld_shared_v4(st + k_chunk_off(g, t + 4));
      const uint4 kB0 = ld_shared_v4(st + k_chunk_off(g + 8, t));
      const uint4 kB1 = ld_shared_v4(st + k_chunk_off(g + 8, t + 4));
      float c[RPW][4];
#pragma unroll
      for (int r = 0; r < RPW; r++) c[r][0] = c[r][1] = c[r][2] = c[r][3] = 0.0f;
#pragma unroll
      for (int cc = 0; cc < 2; cc++)
#pragma unroll
        for (int sub = 0; sub < 4; sub++) {
          const uint32_t wa = word(cc ? kA1 : kA0, sub);
          const uint32_t wb = word(cc ? kB1 : kB0, sub);
          const uint32_t a0 = e4m3_lo2(wa), a2 = e4m3_hi2(wa);
          const uint32_t a1 = e4m3_lo2(wb), a3 = e4m3_hi2(wb);
#pragma unroll
          for (int r = 0; r < RPW; r++)
            mma_f16_16816(c[r], a0, a1, a2, a3, qf[r][4 * cc + sub][0], qf[r][4 * cc + sub][1]);
        }

      // ---- per-key scales; V exponent bookkeeping ----
      const uint32_t ss = st + STAGE_K + STAGE_V;
      const float skg = ld_shared_f32(ss + g * 4), skg8 = ld_shared_f32(ss + (g + 8) * 4);
      const float svg = ld_shared_f32(ss + 64 + g * 4), svg8 = ld_shared_f32(ss + 64 + (g + 8) * 4);
      int be = static_cast<int>(max(__float_as_uint(svg) >> 23, __float_as_uint(svg8) >> 23));
      be = max(be, __shfl_xor_sync(0xffffffffu, be, 4));
      be = max(be, __shfl_xor_sync(0xffffffffu, be, 8));
      be = max(be, __shfl_xor_sync(0xffffffffu, be, 16));
      be = min(be, 253);
      const int bnew = max(bexp, be);
      const float inv = __uint_as_float(static_cast<uint32_t>(254 - bnew) << 23);  // 2^(127-bnew)
      const float sv0 = svg * inv, sv8 = svg8 * inv;
      const float shift = exp2f(static_cast<float>(bexp - bnew));
      bexp = bnew;

      // ---- online softmax (log2 domain), P' = p * scaleV * 2^-E into B fragments of PV ----
      const int64_t jg = jb + g, jg8 = jb + g + 8;
      uint32_t pb0[RPW], pb1[RPW];
#pragma unroll
      for (int r = 0; r < RPW; r++) {
        const int64_t lr = lim[r] < je ? lim[r] : je;
        const float s0 = (jg < lr) ? c[r][0] * (skg * fq[r][0]) : -INFINITY;
        const float s1 = (jg < lr) ? c[r][1] * (skg * fq[r][1]) : -INFINITY;
        const float s2 = (jg8 < lr) ? c[r][2] * (skg8 * fq[r][0]) : -INFINITY;
        const float s3 = (jg8 < lr) ? c[r][3] * (skg8 * fq[r][1]) : -INFINITY;
        float bm0 = fmaxf(s0, s2), bm1 = fmaxf(s1, s3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
          bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
        }
        const float mn0 = fmaxf(m[r][0], bm0), mn1 = fmaxf(m[r][1], bm1);
        const float mu0 = (mn0 == -INFINITY) ? 0.0f : mn0;
        const float mu1 = (mn1 == -INFINITY) ? 0.0f : mn1;
        const float al0 = exp2f(m[r][0] - mu0), al1 = exp2f(m[r][1] - mu1);
        const float p0 = exp2f(s0 - mu0), p1 = exp2f(s1 - mu1);
        const float p2 = exp2f(s2 - mu0), p3 = exp2f(s3 - mu1);
        l[r][0] = l[r][0] * al0 + (p0 + p2);
        l[r][1] = l[r][1] * al1 + (p1 + p3);
        m[r][0] = mn0;
        m[r][1] = mn1;
        const float ac0 = al0 * shift, ac1 = al1 * shift;
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
          acc[r][mt][0] *= ac0;
          acc[r][mt][1] *= ac1;
          acc[r][mt][2] *= ac0;
          acc[r][mt][3] *= ac1;
        }
        pb0[r] = movmatrix_trans(float2_to_f16x2(p0 * sv0, p1 * sv0));   // keys 0..7
        pb1[r] = movmatrix_trans(float2_to_f16x2(p2 * sv8, p3 * sv8));   // keys 8..15
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

  // ---- finalize this warp: full row sums, true numerator scale 2^(E-127) ----
#pragma unroll
  for (int r = 0; r < RPW; r++)
#pragma unroll
    for (int hh = 0; hh < 2; hh++)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) l[r][hh] += __shfl_xor_sync(0xffffffffu, l[r][hh], off);
  const float post = exp2f(static_cast<float>(bexp - 127));

  __syncthreads();  // the rings are free: reuse them as the merge area
  float* merge = reinterpret_cast<float*>(smem);
  if (active) {
#pragma unroll
    for (int r = 0; r < RPW; r++) {
#pragma unroll
      for (int hh = 0; hh < 2; hh++) {
        float* dst = merge + ((warp * RPW + r) * 8 + 2 * t + hh) * MERGE_STRIDE;
        float4* d4 = reinterpret_cast<float4*>(dst + 16 * g);
        // head 2t+hh: d = 16g + 2mt -> acc[mt][hh], d = 16g + 2mt + 1 -> acc[mt][2+hh]
#pragma unroll
        for (int q4 = 0; q4 < 4; q4++)
          d4[q4] = make_float4(acc[r][2 * q4][hh] * post, acc[r][2 * q4][2 + hh] * post,
                               acc[r][2 * q4 + 1][hh] * post, acc[r][2 * q4 + 1][2 + hh] * post);
        if (g == 0) {
          dst[128] = m[r][hh];
          dst[129] = l[r][hh];
        }
      }
    }
  }
  __syncthreads();

  // ---- merge the wk warps of each row group; write this slice's partial ----
  const int items = nrg * RPW * a.group * kHeadDim;
  for (int it = threadIdx.x; it < items; it += blockDim.x) {
    const int d = it % kHeadDim;
    const int hh = (it / kHeadDim) % a.group;
    const int rr = it / (kHeadDim * a.group);      // row index within the request: rg*RPW + r
    if (rr >= R) continue;
    const int rgi = rr / RPW, r = rr % RPW;
    float M = -INFINITY;
    for (int k = 0; k < wk; k++) {
      const float* src = merge + (((rgi * wk + k) * RPW + r) * 8 + hh) * MERGE_STRIDE;
      M = fmaxf(M, src[128]);
    }
    float A = 0.0f, L = 0.0f;
    if (M != -INFINITY) {
      for (int k = 0; k < wk; k++) {
        const float* src = merge + (((rgi * wk + k) * RPW + r) * 8 + hh) * MERGE_STRIDE;
        const float w = exp2f(src[128] - M);
        A += w * src[d];
        L += w * src[129];
      }
    }
    const int64_t prow = ((row0 + rr) * a.num_q_heads + h * a.group + hh) * a.num_splits + split;
    a.part_acc[prow * kHeadDim + d] = A;
    if (d == 0) {
      a.part_ml[prow * 2] = M;
      a.part_ml[prow * 2 + 1] = L;
    }
  }
}

// Merge the slices of one (query row, query head): o = sum_s 2^(M_s-M) A_s / sum_s 2^(M_s-M) L_s.
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeArgs a) {
  const int64_t row = blockIdx.x;
  const int hq = blockIdx.y;
  const int d = threadIdx.x;
  int b;
  if (a.q_row_offsets) {
    int lo = 0, hi = a.batch;  // last b with q_row_offsets[b] <= row
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (a.q_row_offsets[mid] <= row) lo = mid; else hi = mid;
    }
    b = lo;
  } else {
    b = static_cast<int>(row);
  }
  const int64_t n = clamp_seq_len(a, b, false);
  int64_t S = (n + a.chunk - 1) / a.chunk;
  if (S > a.num_splits) S = a.num_splits;
  const int64_t base = (row * a.num_q_heads + hq) * a.num_splits;
  float M = -INFINITY;
  for (int64_t s = 0; s < S; s++) M = fmaxf(M, a.part_ml[(base + s) * 2]);
  float num = 0.0f, den = 0.0f;
  if (M != -INFINITY) {
    for (int64_t s = 0; s < S; s++) {
      const float w = exp2f(a.part_ml[(base + s) * 2] - M);
      num += w * a.part_acc[(base + s) * kHeadDim + d];
      den += w * a.part_ml[(base + s) * 2 + 1];
    }
  }
  const float o = (den > 0.0f) ? num / den : 0.0f;
  a.out[(row * a.num_q_heads + hq) * kHeadDim + d] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
}

template <int RPW>
cudaError_t launch_split(const DecodeArgs& a, cudaStream_t s) {
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<RPW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_bytes<RPW>());
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  dim3 grid(a.num_splits, a.num_kv_heads, a.batch);
  decode_split_kernel<RPW><<<grid, Cfg<RPW>::WARPS * 32, smem_bytes<RPW>(), s>>>(a);
  return cudaGetLastError();
}

}  // namespace

int decode_ctas_per_sm(int max_q_rows) {
  (void)max_q_rows;
  return 1;  // both configurations are shared-memory bound at one CTA per SM
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  cudaError_t e = (a.max_q_rows <= 1) ? launch_split<1>(a, s) : launch_split<2>(a, s);
  if (e != cudaSuccess) return e;
  if (a.total_q_rows > 0) {
    dim3 grid(static_cast<unsigned>(a.total_q_rows), a.num_q_heads);
    decode_combine_kernel<<<grid, 128, 0, s>>>(a);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace ftkv
