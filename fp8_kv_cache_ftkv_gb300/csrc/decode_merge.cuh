// decode_merge.cuh -- the split merge of the decode kernels, run by the CTA whose slice finished last.
//
// Merge of the per-slice partials (FreeToken PR #897, "Fresh R9700 stage-1 A/B": a stage over key
// slices followed by a merge): for each (query row, query head), with per-slice maximum m_s (log2 units),
// sum l_s and unnormalized accumulator O_s,
//     M = max_s m_s,   L = sum_s 2^(m_s - M) l_s,   o = sum_s (2^(m_s - M) / L) O_s      (o = 0 if L = 0).
// The weights are computed by one warp per (row, head) with warp reductions (one thread walking all
// slices three times was a serial tail of microseconds).  The accumulators of one (row, head) are
// contiguous over the slices, and so are their (m, l) pairs: when they fit in the CTA's idle shared
// memory, both arrive by TMA bulk copies (two per (row, head), each pair on its own mbarrier, so merging
// overlaps the copies still in flight); otherwise they are read from L2 with up to 16 loads in flight per
// thread.  (cp.async of every 16 bytes was slower.)
#pragma once

#include "ftkv_device.cuh"
#include "ftkv_internal.h"

namespace ftkv {

__device__ __forceinline__ bool merge_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(100000u)
      : "memory");
  return ok != 0;
}

// Bounded wait for phase 0 of a copy barrier: the copies always complete; the bound (4 s) only guards
// against a fault.  Out of line: it is the cold path of every wait.
static __device__ __noinline__ bool merge_wait_bounded(uint32_t bar) {
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  while (!merge_try_wait(bar, 0)) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > 4000000000ull) return false;
  }
  return true;
}

// w[s] = 2^(m[s] - M) / L for one (row, head), by one warp; wm holds m on entry and the weights on return.
__device__ __forceinline__ void merge_weights_warp(float* wm, const float* wl, int nslices, int lane) {
  float M = -INFINITY;
  for (int sl = lane; sl < nslices; sl += 32) M = fmaxf(M, wm[sl]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float L = 0.0f;
  if (M != -INFINITY)
    for (int sl = lane; sl < nslices; sl += 32) L += exp2f(wm[sl] - M) * wl[sl];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  const float invL = (M != -INFINITY && L > 0.0f) ? 1.0f / L : 0.0f;
  __syncwarp();
  for (int sl = lane; sl < nslices; sl += 32) wm[sl] = (invL != 0.0f) ? exp2f(wm[sl] - M) * invL : 0.0f;
}

// Merge the partials of (request rows row0 .. row0 + nrows - 1, KV head h) into a.out.  buf: the CTA's shared
// memory that is free at this point, at least 8 bytes per (row, head, slice).  Called by every thread.
__device__ __forceinline__ void merge_split_partials(const DecodeArgs& a, int64_t row0, int nrows, int h,
                                                     int nslices, uint8_t* buf, uint32_t buf_bytes) {
  const int G = a.group;
  const int npairs = nrows * G;  // pair pr = (row pr / G, head pr % G)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int64_t pstride = static_cast<int64_t>(a.num_splits) * a.pps;  // partial slots per (row, head)
  auto prow0 = [&](int pr) -> int64_t {  // partial row of (pair pr, slice 0)
    return ((row0 + pr / G) * a.num_q_heads + h * G + pr % G) * pstride;
  };
  // Bulk path (even slice counts keep every copy a multiple of 16 bytes and 16-byte aligned): per (row, head),
  // one copy of its nslices x 128 accumulators and one of its nslices (m, l) pairs, completing on that pair's
  // own mbarrier, so a pair is merged as soon as its data has landed while later pairs are still in flight.
  // Two warps take one pair: weights from shared memory with one exp2 per slice (each warp its own copy),
  // then the 32 x 4 outputs, even and odd slices on adjacent lanes.
  const uint32_t acc_bytes = static_cast<uint32_t>(npairs) * nslices * kHeadDim * 4;
  const uint32_t ml_bytes = static_cast<uint32_t>(npairs) * nslices * 8;
  const uint32_t wgt_bytes = static_cast<uint32_t>(nwarps) * 64 * 4;
  // (m, l) copies start at part_ml + 8 prow0 bytes, prow0 a multiple of the slot count per (row, head): 16-byte
  // aligned when that count is even; the accumulator copies start at 512 prow0 bytes.
  const bool bulk = (nslices % 2 == 0) && (pstride % 2 == 0) && nslices <= 64 && (nwarps % 2 == 0) &&
                    static_cast<uint64_t>(acc_bytes) + ml_bytes + wgt_bytes + 8ull * npairs <= buf_bytes;
  if (bulk) {
    const float* pacc = reinterpret_cast<const float*>(buf);              // [npairs][nslices][128]
    const float* pml = reinterpret_cast<const float*>(buf + acc_bytes);   // [npairs][nslices][2]
    float* wgt = reinterpret_cast<float*>(buf + acc_bytes + ml_bytes);    // [nwarps][64]
    const uint32_t mbar0 = smem_addr(buf) + acc_bytes + ml_bytes + wgt_bytes;  // [npairs] x 8 bytes
    const uint32_t per = static_cast<uint32_t>(nslices) * kHeadDim * 4, per_ml = static_cast<uint32_t>(nslices) * 8;
    // earlier generic accesses to the buffer come before the async proxy overwrites it
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int pr = 0; pr < npairs; pr++)
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbar0 + 8 * pr) : "memory");
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();  // every barrier is initialised before any thread polls it
    if (threadIdx.x == 0) {
      // the other slices' partials were written by generic stores, released through the ticket
      asm volatile("fence.proxy.async.global;" ::: "memory");
      for (int pr = 0; pr < npairs; pr++) {
        const uint32_t mb = mbar0 + 8 * pr;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb), "r"(per + per_ml) : "memory");
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                smem_addr(buf) + pr * per),
            "l"(a.part_acc + prow0(pr) * kHeadDim), "r"(per), "r"(mb)
            : "memory");
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                smem_addr(buf) + acc_bytes + pr * per_ml),
            "l"(a.part_ml + prow0(pr) * 2), "r"(per_ml), "r"(mb)
            : "memory");
      }
    }
    float* wm = wgt + warp * 64;
    for (int pr = warp >> 1; pr < npairs; pr += nwarps >> 1) {  // warp-uniform
      // bounded wait for this pair's copies (they always complete; the bound only guards against a fault)
      const uint32_t mb = mbar0 + 8 * pr;
      const bool landed = merge_try_wait(mb, 0) || merge_wait_bounded(mb);
      if (!__all_sync(0xffffffffu, landed)) {
        if (lane == 0) flag_error(a.err, kDevErrTimeout);
        break;
      }
      // weights of this pair: lanes take slices lane and lane + 32
      const float* ml = pml + pr * nslices * 2;
      const bool h0 = lane < nslices, h1 = lane + 32 < nslices;
      const float m0 = h0 ? ml[2 * lane] : -INFINITY, m1 = h1 ? ml[2 * (lane + 32)] : -INFINITY;
      float M = fmaxf(m0, m1);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
      const float e0 = (h0 && M != -INFINITY) ? exp2f(m0 - M) : 0.0f;
      const float e1 = (h1 && M != -INFINITY) ? exp2f(m1 - M) : 0.0f;
      float L = (h0 ? e0 * ml[2 * lane + 1] : 0.0f) + (h1 ? e1 * ml[2 * (lane + 32) + 1] : 0.0f);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
      const float invL = (M != -INFINITY && L > 0.0f) ? 1.0f / L : 0.0f;
      if (h0) wm[lane] = e0 * invL;
      if (h1) wm[lane + 32] = e1 * invL;
      __syncwarp();
      // o = sum_s w_s O_s over this lane's slice parity; the two parities meet through one shuffle
      const int item = (warp & 1) * 32 + lane;  // (4 d values, slice parity) of the pair
      const int part = item & 1, d4 = item >> 1;
      const float4* src = reinterpret_cast<const float4*>(pacc + static_cast<int64_t>(pr) * nslices * kHeadDim) + d4;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int sl = part; sl < nslices; sl += 2) {
        const float4 v = src[sl * (kHeadDim / 4)];
        const float wv = wm[sl];
        o.x += wv * v.x;
        o.y += wv * v.y;
        o.z += wv * v.z;
        o.w += wv * v.w;
      }
      o.x += __shfl_xor_sync(0xffffffffu, o.x, 1);
      o.y += __shfl_xor_sync(0xffffffffu, o.y, 1);
      o.z += __shfl_xor_sync(0xffffffffu, o.z, 1);
      o.w += __shfl_xor_sync(0xffffffffu, o.w, 1);
      if (part == 0) {
        const uint2 packed = make_uint2(float2_to_bf16x2(o.x, o.y), float2_to_bf16x2(o.z, o.w));
        *reinterpret_cast<uint2*>(a.out + ((row0 + pr / G) * a.num_q_heads + h * G + pr % G) * kHeadDim + 4 * d4) =
            packed;
      }
      __syncwarp();  // the weights are rewritten for the next pair
    }
    return;
  }
  // L2 path, in chunks of pairs whose (m, l) fit in the buffer: [2][np][nslices], m then l, m replaced by the
  // weights.
  const int chunk_pairs = static_cast<int>(buf_bytes / (8u * static_cast<uint32_t>(nslices))) > 0
                              ? static_cast<int>(buf_bytes / (8u * static_cast<uint32_t>(nslices)))
                              : 1;
  for (int pc = 0; pc < npairs; pc += chunk_pairs) {
    const int np = (npairs - pc < chunk_pairs) ? npairs - pc : chunk_pairs;
    float* wts = reinterpret_cast<float*>(buf);
    __syncthreads();  // the previous chunk is done with the buffer
    for (int i = threadIdx.x; i < np * nslices; i += blockDim.x) {
      const int pr = pc + i / nslices, sl = i % nslices;
      const int64_t p = prow0(pr) + sl;
      wts[i] = __ldcg(a.part_ml + p * 2);
      wts[np * nslices + i] = __ldcg(a.part_ml + p * 2 + 1);
    }
    __syncthreads();
    for (int q = warp; q < np; q += nwarps)
      merge_weights_warp(wts + q * nslices, wts + np * nslices + q * nslices, nslices, lane);
    __syncthreads();
    // Output: item (pair, 4 d values) split over 2 adjacent lanes, each summing every other slice with up to 16
    // loads in flight; the two halves meet through one shuffle.  np * 64 and blockDim.x are multiples of 32, so
    // every warp is either fully inside the range or fully outside it.
    constexpr int SPLIT = 2, BATCH = 16;
    const int total = np * (kHeadDim / 4) * SPLIT;
    for (int it = threadIdx.x; it < total; it += blockDim.x) {
      const int part = it % SPLIT, item = it / SPLIT;
      const int d4 = item % (kHeadDim / 4), q = item / (kHeadDim / 4), pr = pc + q;
      const float* wm = wts + q * nslices;
      const float4* src = reinterpret_cast<const float4*>(a.part_acc + prow0(pr) * kHeadDim) + d4;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s0 = part; s0 < nslices; s0 += SPLIT * BATCH) {
        float4 v[BATCH];
#pragma unroll
        for (int u = 0; u < BATCH; u++) {
          const int sl = s0 + SPLIT * u;
          v[u] = (sl < nslices) ? __ldcg(src + static_cast<int64_t>(sl) * (kHeadDim / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < BATCH; u++) {
          const int sl = s0 + SPLIT * u;
          const float wv = (sl < nslices) ? wm[sl] : 0.0f;
          o.x += wv * v[u].x;
          o.y += wv * v[u].y;
          o.z += wv * v[u].z;
          o.w += wv * v[u].w;
        }
      }
#pragma unroll
      for (int off = 1; off < SPLIT; off <<= 1) {
        o.x += __shfl_xor_sync(0xffffffffu, o.x, off);
        o.y += __shfl_xor_sync(0xffffffffu, o.y, off);
        o.z += __shfl_xor_sync(0xffffffffu, o.z, off);
        o.w += __shfl_xor_sync(0xffffffffu, o.w, off);
      }
      if (part == 0) {
        const uint2 packed = make_uint2(float2_to_bf16x2(o.x, o.y), float2_to_bf16x2(o.z, o.w));
        *reinterpret_cast<uint2*>(a.out + ((row0 + pr / G) * a.num_q_heads + h * G + pr % G) * kHeadDim + 4 * d4) =
            packed;
      }
    }
  }
}

}  // namespace ftkv
