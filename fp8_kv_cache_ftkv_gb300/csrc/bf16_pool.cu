// bf16_pool.cu -- the unquantized comparison point: decode attention and the prefix gather over a BF16 KV pool.
//
// FreeToken keeps BF16 KV as its default ("KV_FMT none" in the kernel variants of PR #897, opening description;
// PR #853, "What changes": FP8 is opt-in), and the pages weigh FP8 against it by bytes per token (98,304 vs
// 50,688 at their model's geometry, PR #853 "Validation") and by decode and prefill speed.  These kernels are
// that BF16 path on this GPU, so that the two formats can be timed side by side:
//  * decode: for query row r of request b (R rows, n keys), per query head i (KV head h = i / G),
//        s_j = (q . k_j) * sm_scale,  o = sum_j softmax(s)_j v_j,   over the row's visible keys
//    (causal within the new rows, optionally a sliding window), with the split-K geometry, partial layout and
//    split merge of the FP8 decode (decode_common.cuh), so its results are directly comparable;
//  * prefill: the historical rows are gathered from the pool into the shared BF16 workspace in logical order
//    (the BF16 counterpart of the FP8 reconstruction, PR #853 "What changes"), after which the same prefill
//    kernel runs over it.
//
// Decode design (the FP8 single-row kernel's structure with BF16 operands):
//  * A CTA covers one key slice of one query row for HC (up to 4) KV heads: a token's K (and V) rows for those
//    heads are one contiguous run of HC x 256 bytes, copied with 16-byte cp.async by whole warps.
//  * 4 warps in NG = 4 / HC key groups of HC warps (one per KV head); a group shares a 3-stage ring of
//    16-key blocks; the groups' partials are combined in shared memory at the end, so a key slice yields one
//    partial.  96 KB of ring plus the slot window: two CTAs per SM.
//  * Per 16-key block and warp: S^T = K Q^T on BF16 tensor cores (keys as M, the KV head's 8 query heads as
//    N; K fragments by ldmatrix from an XOR-swizzled stage), a softmax with a lazy running maximum, then
//    O^T += V^T P^T (V^T fragments by ldmatrix.trans, P transposed with movmatrix).  The MMA's A and B share
//    one type and V is BF16, so P enters as two BF16 pieces, P = hi + lo (16 significant bits), in two MMAs:
//    with P in BF16 alone, an output element small next to the terms it sums would be off by up to 2^-9 of
//    those terms.
//  * Multi-row batches: each query row runs as its own set of CTAs over the request's key slices (every row
//    re-reads the keys it sees; the FP8 multi-row kernel shares them).  A slice outside a row's visible range
//    publishes an empty partial.
//  * Fused store (k_new / v_new given): new tokens are read straight from k_new / v_new, and the CTA whose
//    slice holds a row's own token copies that token's rows into the pool.
#include <climits>
#include <mutex>

#include "decode_common.cuh"
#include "ftkv_device.cuh"
#include "ftkv_internal.h"

namespace ftkv {
namespace {

constexpr int BW = 4;       // warps per CTA
constexpr int BKB = 16;     // keys per block
constexpr int BNS = 3;      // ring stages per key group
constexpr int BWIN = 1024;  // slot indices staged in shared memory at a time
constexpr float kLazyMaxB = 8.0f;  // log2 slack of the running maximum

template <int HC>
struct Bf {
  static constexpr int NG = BW / HC;                   // key groups
  static constexpr int RUN = HC * kHeadDim * 2;        // bytes of one token's K (or V) rows for the HC heads
  static constexpr int V_OFF = BKB * RUN;              // stage: K runs [16][RUN], V runs [16][RUN]
  static constexpr int STAGE = 2 * BKB * RUN;
  static constexpr int RING = NG * BNS * STAGE;
  static constexpr int SLOT_OFF = RING;                // [BWIN] int32 slot indices
  static constexpr int SMEM = SLOT_OFF + BWIN * 4;
};
static_assert(Bf<4>::SMEM <= 113 * 1024 && Bf<2>::SMEM <= 113 * 1024 && Bf<1>::SMEM <= 113 * 1024,
              "two CTAs per SM");

// Shared-memory offset of 16-byte chunk p (d = 8p .. 8p+7) of KV head hd of key `key` (0..15) within a stage
// half.  The XOR with key & 7 makes the 8 rows of every ldmatrix phase, and the cp.async run writes, free of
// bank conflicts.
template <int HC>
__device__ __forceinline__ uint32_t bf_off(int key, int hd, int p) {
  return key * Bf<HC>::RUN + hd * (kHeadDim * 2) + ((p ^ (key & 7)) << 4);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr) : "memory");
}

template <int HC>
__global__ void __launch_bounds__(BW * 32, 2) decode_bf16_kernel(const DecodeArgs a) {
  using T = Bf<HC>;
  constexpr int NG = T::NG;
  extern __shared__ __align__(128) uint8_t smem[];
  int32_t* sslot = reinterpret_cast<int32_t*>(smem + T::SLOT_OFF);
  griddep_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = warp / HC, hh = warp % HC;  // key group; KV head of this warp within the CTA
  const int lt = hh * 32 + lane;             // thread within the group
  const int g = lane >> 2, t = lane & 3;
  const int split = blockIdx.x, h0 = blockIdx.y * HC;
  const int64_t row = blockIdx.z;            // query row
  const int hkv = a.num_kv_heads;
  const int64_t tok_stride = static_cast<int64_t>(hkv) * kHeadDim;  // elements of one pool row
  const uint32_t ring = smem_addr(smem) + gi * BNS * T::STAGE;

  // ---- the row's request.  Without row offsets the row is the request, and under the stable-history
  // contract the slot table, the lengths and the history rows may be read before the preceding grid ends ----
  const bool early = a.early && !a.q_row_offsets;
  if (!early) griddep_wait();
  int b = static_cast<int>(row), R = 1;
  int64_t row0 = row;
  bool bad_rows = false;
  if (a.q_row_offsets) {
    int lo = 0, hi = a.batch;  // the merge's search, so both sides agree on the request
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (a.q_row_offsets[mid + 1] <= row) lo = mid + 1; else hi = mid;
    }
    b = lo;
    if (b >= a.batch) {
      bad_rows = true;
      b = 0;
    } else {
      row0 = a.q_row_offsets[b];
      R = a.q_row_offsets[b + 1] - a.q_row_offsets[b];
      bad_rows = R < 0 || R > a.max_q_rows || row0 < 0 || row0 + R > a.total_q_rows || row < row0 || row >= row0 + R;
    }
  }
  if (bad_rows) {
    if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) flag_error(a.err, kDevErrQRows);
    if (a.coop) coop_finish<BW>(a);
    return;
  }
  const int r = static_cast<int>(row - row0);
  const int64_t n = clamp_seq_len(a, b, threadIdx.x == 0 && split == 0 && blockIdx.y == 0 && r == 0);

  // ---- key ranges: the slice [j0, j1) of the request's attended keys, and this row's part [ks, ke) of it ----
  const int j0 = static_cast<int>(first_key(a, n, R)) + split * static_cast<int>(a.chunk);  // 32-bit (host check)
  const int j1 = (static_cast<int64_t>(j0) + a.chunk < n) ? j0 + static_cast<int>(a.chunk) : static_cast<int>(n);
  if (j0 >= j1) {  // the slice holds no key of the request: nothing to publish (the merge does not read it)
    if (early) griddep_wait();
    if (a.coop) coop_finish<BW>(a);
    return;
  }
  const int vis = static_cast<int>(n) - R + r + 1;  // keys 0 .. vis-1 are visible to this row
  const int low = (a.window > 0 && vis - a.window > 0) ? vis - static_cast<int>(a.window) : 0;
  const int ks = j0 > low ? j0 : low;
  const int ke = j1 < vis ? j1 : vis;  // ks >= ke: an empty partial
  const int new_lo = a.k_new ? static_cast<int>(n) - R : INT_MAX;  // positions >= new_lo are the new tokens
  const int hist_end = static_cast<int>(n) - a.max_q_rows;           // keys below are history

  // ---- per-thread load plan: every block, this thread copies chunk ld_p of KV head ld_hd of keys
  // kr, kr + 2, .., kr + 14, of K and of V ----
  const int ck = lt % (16 * HC), kr = lt / (16 * HC);
  const int ld_hd = ck >> 4, ld_p = ck & 15;
  const int64_t goff = (h0 + ld_hd) * kHeadDim + ld_p * 8;
  const uint64_t pol = l2_policy_evict_first();  // the key loop reads every line once

  auto stage_slots = [&](int js, int nk) {
    for (int i = threadIdx.x; i < nk; i += blockDim.x) {
      int32_t sv = a.req_to_slot[static_cast<int64_t>(b) * a.req_stride + js + i];
      if (js + i < new_lo && (sv < 0 || sv >= a.num_rows)) {  // new tokens come from k_new / v_new
        flag_error(a.err, kDevErrBadSlot);
        sv = 0;
      }
      sslot[i] = sv;
    }
  };
  // Block i of this group within the window [js, js + nk): keys js + (gi + i NG) 16 .. +15, into stage i % BNS.
  // Keys past the window are zero-filled (a zero V row keeps the masked products finite).
  auto issue = [&](int i, int my_nblk, int js, int nk) {
    if (i < my_nblk) {
      const int key0 = (gi + i * NG) * BKB;
      const uint32_t st = ring + (i % BNS) * T::STAGE;
#pragma unroll
      for (int u = 0; u < 8; u++) {
        const int kb = kr + 2 * u;
        const uint32_t dk = st + bf_off<HC>(kb, ld_hd, ld_p);
        const int key = key0 + kb;
        if (key < nk) {
          const int pos = js + key;
          const uint16_t *sk, *sv;
          if (pos >= new_lo) {  // a new token: its rows come from k_new / v_new (row row0 + pos - new_lo)
            const int64_t o = (row0 + pos - new_lo) * tok_stride + goff;
            sk = a.k_new + o;
            sv = a.v_new + o;
          } else {
            const int64_t o = static_cast<int64_t>(sslot[key]) * tok_stride + goff;
            sk = a.k_bf16 + o;
            sv = a.v_bf16 + o;
          }
          cp_async_16_hint(dk, sk, pol);
          cp_async_16_hint(dk + T::V_OFF, sv, pol);
        } else {
          st_shared_zero16(dk);
          st_shared_zero16(dk + T::V_OFF);
        }
      }
    }
    cp_async_commit();
  };
  auto window_blocks = [&](int nk) {  // this group's blocks in a window of nk keys
    const int nblk = (nk + BKB - 1) / BKB;
    return nblk > gi ? (nblk - gi + NG - 1) / NG : 0;
  };

  const int nk0 = ks < ke ? ((ke - ks < BWIN) ? ke - ks : BWIN) : 0;
  int pre = 0;  // blocks of the first window issued before the wait
  if (early) {  // history blocks before the wait (contract), then the wait
    if (nk0 > 0) stage_slots(ks, nk0);
    __syncthreads();
    const int mb0 = window_blocks(nk0);
    for (int i = 0; i < BNS; i++) {  // group-uniform
      if (i >= mb0 || ks + (gi + i * NG) * BKB + BKB > hist_end) break;
      issue(i, mb0, ks, nk0);
      pre = i + 1;
    }
    griddep_wait();
  } else if (nk0 > 0) {
    stage_slots(ks, nk0);
  }

  // ---- fused store of this row's own token (position n - R + r), by the CTA whose slice holds it: one warp
  // per KV head, K row on lanes 0-15 and V row on lanes 16-31 ----
  const int my_pos = static_cast<int>(n) - R + r;
  if (a.k_new && my_pos >= j0 && my_pos < j1 && warp < HC) {
    const int half = lane >> 4, l16 = lane & 15;
    const int64_t src = row * tok_stride + (h0 + warp) * kHeadDim + l16 * 8;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>((half ? a.v_new : a.k_new) + src));
    const int32_t sv = a.req_to_slot[static_cast<int64_t>(b) * a.req_stride + my_pos];
    if (sv >= 0 && sv < a.num_rows) {
      // the pool is the caller's writable memory; this kernel reads new tokens from k_new / v_new only
      uint16_t* dst = const_cast<uint16_t*>(half ? a.v_bf16 : a.k_bf16);
      *reinterpret_cast<uint4*>(dst + static_cast<int64_t>(sv) * tok_stride + (h0 + warp) * kHeadDim + l16 * 8) = v;
    } else if (lane == 0) {
      flag_error(a.err, kDevErrBadSlot);
    }
  }

  // ---- B operand of QK^T: query head g of this warp's KV head, d = 16kk + 2t (+1) and 16kk + 2t + 8 (+9) ----
  const int G = a.group;
  uint32_t qb[8][2];
  {
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(
        a.q + (row * a.num_q_heads + (h0 + hh) * G + (g < G ? g : 0)) * kHeadDim);
#pragma unroll
    for (int kk = 0; kk < 8; kk++) {
      qb[kk][0] = g < G ? __ldg(q32 + 8 * kk + t) : 0u;
      qb[kk][1] = g < G ? __ldg(q32 + 8 * kk + t + 4) : 0u;
    }
  }
  __syncthreads();  // the slot window is staged

  // ldmatrix row addresses (lane-dependent parts): K fragments take keys (lane & 7) + 8 ((lane >> 3) & 1) at
  // chunk 2kk + (lane >> 4); V^T fragments keys (lane & 7) + 8 (lane >> 4) at chunk 2mt + ((lane >> 3) & 1)
  const int kkey = (lane & 7) + (((lane >> 3) & 1) << 3), khi = lane >> 4;
  const int vkey = (lane & 7) + ((lane >> 4) << 3), vhi = (lane >> 3) & 1;

  float acc[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; mt++) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.0f;
  float m[2] = {-INFINITY, -INFINITY};  // running maximum of s (log2 units), query heads 2t, 2t+1
  float l[2] = {0.0f, 0.0f};            // this lane's share of sum 2^(s - m)
  const float qs = a.qk_scale_log2;

  for (int js = ks; js < ke; js += BWIN) {  // CTA-uniform
    const int je = (js + BWIN < ke) ? js + BWIN : ke;
    const int nk = je - js;
    int done = 0;
    if (js == ks) {
      done = pre;
    } else {
      __syncthreads();  // every group is done with the previous window's slots and stages
      stage_slots(js, nk);
      __syncthreads();
    }
    const int my_nblk = window_blocks(nk);
    for (int i = done; i < BNS; i++) issue(i, my_nblk, js, nk);

#pragma unroll 1
    for (int i = 0; i < my_nblk; i++) {
      if (i == 0) cp_async_wait<BNS - 1>(); else cp_async_wait<BNS - 2>();
      group_barrier<NG>(gi, 32 * HC);  // block i landed for every thread; block i - 1 is free
      if (i > 0) issue(i + BNS - 1, my_nblk, js, nk);
      const uint32_t st = ring + (i % BNS) * T::STAGE;
      const int jb = js + (gi + i * NG) * BKB;

      // ---- S^T = K Q^T: keys as M (rows g, g+8), query heads as N, d as K in 8 steps of 16 ----
      float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int kk = 0; kk < 8; kk++) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(st + bf_off<HC>(kkey, hh, 2 * kk + khi), a0, a1, a2, a3);
        mma_bf16_16816(c, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
      }

      // ---- softmax with a lazy maximum (log2 domain) ----
      const bool in0 = jb + g < je, in8 = jb + g + 8 < je;
      const float s0 = in0 ? c[0] * qs : -INFINITY, s1 = in0 ? c[1] * qs : -INFINITY;
      const float s2 = in8 ? c[2] * qs : -INFINITY, s3 = in8 ? c[3] * qs : -INFINITY;
      const bool raise = fmaxf(s0, s2) > m[0] + kLazyMaxB || fmaxf(s1, s3) > m[1] + kLazyMaxB;
      if (__any_sync(0xffffffffu, raise)) {  // new maximum: exact block max, rescale
        float bm0 = fmaxf(s0, s2), bm1 = fmaxf(s1, s3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
          bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
        }
        const float mn0 = fmaxf(m[0], bm0), mn1 = fmaxf(m[1], bm1);
        const float al0 = (m[0] == -INFINITY) ? 1.0f : fast_exp2(m[0] - mn0);
        const float al1 = (m[1] == -INFINITY) ? 1.0f : fast_exp2(m[1] - mn1);
        m[0] = mn0;
        m[1] = mn1;
        l[0] *= al0;
        l[1] *= al1;
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
          acc[mt][0] *= al0;
          acc[mt][1] *= al1;
          acc[mt][2] *= al0;
          acc[mt][3] *= al1;
        }
      }
      const float mu0 = (m[0] == -INFINITY) ? 0.0f : m[0], mu1 = (m[1] == -INFINITY) ? 0.0f : m[1];
      const float p0 = fast_exp2(s0 - mu0), p1 = fast_exp2(s1 - mu1);
      const float p2 = fast_exp2(s2 - mu0), p3 = fast_exp2(s3 - mu1);
      l[0] += p0 + p2;
      l[1] += p1 + p3;
      // P = hi + lo in BF16 (lo: the rounding residual of hi, itself rounded)
      const uint32_t hk0 = float2_to_bf16x2(p0, p1), hk1 = float2_to_bf16x2(p2, p3);  // keys g, g + 8
      const uint32_t lk0 = float2_to_bf16x2(p0 - bf16_lo(hk0), p1 - bf16_hi(hk0));
      const uint32_t lk1 = float2_to_bf16x2(p2 - bf16_lo(hk1), p3 - bf16_hi(hk1));
      const uint32_t hb0 = movmatrix_trans(hk0), hb1 = movmatrix_trans(hk1);
      const uint32_t lb0 = movmatrix_trans(lk0), lb1 = movmatrix_trans(lk1);

      // ---- O^T += V^T P^T: d as M (d = 16mt + g, + 8), query heads as N, keys as K ----
#pragma unroll
      for (int mt = 0; mt < 8; mt++) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(st + T::V_OFF + bf_off<HC>(vkey, hh, 2 * mt + vhi), a0, a1, a2, a3);
        mma_bf16_16816(acc[mt], a0, a1, a2, a3, hb0, hb1);
        mma_bf16_16816(acc[mt], a0, a1, a2, a3, lb0, lb1);
      }
    }
    cp_async_wait<0>();
  }

  // ---- one partial per (row, query head) and key slice: groups 1 .. NG-1 leave m, l and the accumulator in the
  // ring area, group 0 folds them into its own and writes the result in the transposed layout ----
#pragma unroll
  for (int hx = 0; hx < 2; hx++)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) l[hx] += __shfl_xor_sync(0xffffffffu, l[hx], off);
  const int64_t nsl = a.num_splits;  // one partial per slice (pps = 1)
  if constexpr (NG > 1) {
    float* gacc = reinterpret_cast<float*>(smem);                   // [NG-1][HC][8][128]
    float* gml = gacc + (NG - 1) * HC * 8 * kHeadDim;               // [NG-1][HC][8][2]
    __syncthreads();  // every group is done with the ring
    if (gi > 0) {
#pragma unroll
      for (int hx = 0; hx < 2; hx++) {
        float* dst = gacc + (((gi - 1) * HC + hh) * 8 + 2 * t + hx) * kHeadDim;
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
          dst[16 * mt + g] = acc[mt][hx];
          dst[16 * mt + g + 8] = acc[mt][2 + hx];
        }
        if (g == 0) *reinterpret_cast<float2*>(gml + (((gi - 1) * HC + hh) * 8 + 2 * t + hx) * 2) = make_float2(m[hx], l[hx]);
      }
    }
    __syncthreads();
#pragma unroll 1
    for (int go = 1; go < NG && gi == 0; go++) {
#pragma unroll
      for (int hx = 0; hx < 2; hx++) {
        const int slot = ((go - 1) * HC + hh) * 8 + 2 * t + hx;
        const float2 mlo = *reinterpret_cast<const float2*>(gml + slot * 2);
        const float mn = fmaxf(m[hx], mlo.x);
        if (mn == -INFINITY) continue;  // neither holds a key
        const float f = (m[hx] == -INFINITY) ? 0.0f : fast_exp2(m[hx] - mn);
        const float fo = (mlo.x == -INFINITY) ? 0.0f : fast_exp2(mlo.x - mn);
        const float* src = gacc + slot * kHeadDim;
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
          acc[mt][hx] = fmaf(acc[mt][hx], f, src[16 * mt + g] * fo);
          acc[mt][2 + hx] = fmaf(acc[mt][2 + hx], f, src[16 * mt + g + 8] * fo);
        }
        l[hx] = fmaf(l[hx], f, mlo.y * fo);
        m[hx] = mn;
      }
    }
  }
#pragma unroll
  for (int hx = 0; hx < 2; hx++) {
    const int hq = 2 * t + hx;
    if (gi == 0 && hq < G) {
      const int64_t prow = row * a.num_q_heads + (h0 + hh) * G + hq;
      float* dst = a.part_acc + prow * kHeadDim * nsl;  // element d of slice s at ((d / 4) nsl + s) 4 + d % 4
#pragma unroll
      for (int mt = 0; mt < 8; mt++) {
        const int d0 = 16 * mt + g, d1 = d0 + 8;
        dst[((d0 >> 2) * nsl + split) * 4 + (d0 & 3)] = acc[mt][hx];
        dst[((d1 >> 2) * nsl + split) * 4 + (d1 & 3)] = acc[mt][2 + hx];
      }
      if (g == 0) *reinterpret_cast<float2*>(a.part_ml + (prow * nsl + split) * 2) = make_float2(m[hx], l[hx]);
    }
  }
  if (a.coop) coop_finish<BW>(a);
}

template <int HC>
cudaError_t launch_bf16(const DecodeArgs& a, cudaStream_t s, int dev) {
  static std::once_flag once[kMaxDecodeDevices];
  static cudaError_t setup_err[kMaxDecodeDevices];
  static int resident[kMaxDecodeDevices];
  std::call_once(once[dev], [&] {
    setup_err[dev] = cudaFuncSetAttribute(decode_bf16_kernel<HC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          Bf<HC>::SMEM);
    int coop_ok = 0, sms = 0, per_sm = 0;
    if (setup_err[dev] == cudaSuccess) setup_err[dev] = cudaDeviceGetAttribute(&coop_ok, cudaDevAttrCooperativeLaunch, dev);
    if (setup_err[dev] == cudaSuccess) setup_err[dev] = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (setup_err[dev] == cudaSuccess &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_bf16_kernel<HC>, BW * 32, Bf<HC>::SMEM) !=
            cudaSuccess)
      per_sm = 0;
    resident[dev] = (coop_ok && per_sm > 0 && sms > 0) ? per_sm * sms : -1;
  });
  if (setup_err[dev] != cudaSuccess) return setup_err[dev];
  const dim3 grid(a.num_splits, a.num_kv_heads / HC, static_cast<unsigned>(a.total_q_rows));
  DecodeArgs c = a;
  c.pps = 1;
  c.ptrans = 1;
  const int64_t ctas = int64_t(grid.x) * grid.y * grid.z;
  c.coop = (resident[dev] > 0 && ctas <= resident[dev]) ? 1 : 0;
  if (c.coop) return launch_k_coop(decode_bf16_kernel<HC>, grid, dim3(BW * 32), Bf<HC>::SMEM, s, c);
  cudaError_t e = launch_k(decode_bf16_kernel<HC>, grid, dim3(BW * 32), Bf<HC>::SMEM, s, c);
  if (e != cudaSuccess) return e;
  const int64_t items = a.total_q_rows * a.num_q_heads * (kHeadDim / 4);
  return launch_k(decode_merge_kernel<kMergeWarps>, dim3(static_cast<unsigned>((items + kMergeWarps - 1) / kMergeWarps)),
                  dim3(kMergeWarps * 32), 0, s, c);
}

// ---- prefix gather: ws[i][h][:] = pool[slots[i]][h][:] for K and V; 16 lanes per (row, head) unit, GU units
// per lane group with every load in flight before the stores; a slot outside the pool is flagged and its
// workspace row written as zeros ----
constexpr int GU = 4;
__global__ void __launch_bounds__(256) gather_bf16_kernel(GatherArgs a) {
  pdl_enter();
  const int64_t grp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 4;
  const int l = threadIdx.x & 15;
  const int64_t total = a.num_prefix * a.num_kv_heads;
  uint4 kv[GU], vv[GU];
#pragma unroll
  for (int u = 0; u < GU; u++) {
    const int64_t unit = grp * GU + u;  // unit = i * Hkv + h
    const int64_t i = unit / a.num_kv_heads;
    const int h = static_cast<int>(unit - i * a.num_kv_heads);
    const int32_t sv = unit < total ? __ldg(a.slots + i) : -1;
    const bool ok = sv >= 0 && sv < a.num_rows;
    if (unit < total && !ok && l == 0) flag_error(a.err, kDevErrBadSlot);
    const int64_t off = (static_cast<int64_t>(sv) * a.num_kv_heads + h) * kHeadDim + l * 8;
    kv[u] = ok ? ldg_stream16(a.k + off) : make_uint4(0u, 0u, 0u, 0u);
    vv[u] = ok ? ldg_stream16(a.v + off) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int u = 0; u < GU; u++) {
    const int64_t unit = grp * GU + u;
    if (unit >= total) break;
    reinterpret_cast<uint4*>(a.ws_k + unit * kHeadDim)[l] = kv[u];
    reinterpret_cast<uint4*>(a.ws_v + unit * kHeadDim)[l] = vv[u];
  }
}

}  // namespace

cudaError_t launch_decode_bf16(const DecodeArgs& a, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDecodeDevices) return cudaErrorInvalidDevice;
  switch (decode_tok_heads_per_cta(a.num_kv_heads)) {
    case 4: return launch_bf16<4>(a, s, dev);
    case 2: return launch_bf16<2>(a, s, dev);
    default: return launch_bf16<1>(a, s, dev);
  }
}

cudaError_t launch_gather_bf16(const GatherArgs& a, cudaStream_t s) {
  const int64_t groups = (a.num_prefix * a.num_kv_heads + GU - 1) / GU;
  const int64_t blocks = (groups * 16 + 255) / 256;
  return launch_k(gather_bf16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, a);
}

}  // namespace ftkv
