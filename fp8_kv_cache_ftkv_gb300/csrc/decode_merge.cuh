// decode_merge.cuh -- the split merge of the decode kernels, run by the CTA whose slice finished last.
//
// Merge of the per-slice partials (FreeToken PR #897, "Fresh R9700 stage-1 A/B": a stage over key
// slices followed by a merge): for each (query row, query head), with per-slice maximum m_s (log2 units),
// sum l_s and unnormalized accumulator O_s,
//     M = max_s m_s,   L = sum_s 2^(m_s - M) l_s,   o = sum_s (2^(m_s - M) / L) O_s      (o = 0 if L = 0).
// The weights are computed by one warp per (row, head) with warp reductions (one thread walking all
// slices three times was a serial tail of microseconds); the accumulators are read from L2 with up to 16
// loads in flight per thread.  (Copying all partials into shared memory first with cp.async was slower.)
#pragma once

#include "ftkv_device.cuh"
#include "ftkv_internal.h"

namespace ftkv {

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
                                                     int nslices, uint8_t* buf) {
  const int G = a.group;
  const int npairs = nrows * G;  // pair pr = (row pr / G, head pr % G)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  auto prow0 = [&](int pr) -> int64_t {  // partial row of (pair pr, slice 0)
    return ((row0 + pr / G) * a.num_q_heads + h * G + pr % G) * a.num_splits;
  };
  float* wts = reinterpret_cast<float*>(buf);  // [2][npairs][nslices]: m then l, m replaced by the weights
  // Output: item (pair, 4 d values) split over 2 adjacent lanes, each summing every other slice with up to 16
  // loads in flight; the two halves meet through one shuffle.  npairs * 64 and blockDim.x are multiples
  // of 32, so every warp is either fully inside the range or fully outside it.  (Loading the first batch
  // before the weights overlapped one round trip but made both kernels spill: slower overall.)
  constexpr int SPLIT = 2, BATCH = 16;
  const int total = npairs * (kHeadDim / 4) * SPLIT;
  auto acc_src = [&](int it) {
    const int item = it / SPLIT, d4 = item % (kHeadDim / 4), pr = item / (kHeadDim / 4);
    return reinterpret_cast<const float4*>(a.part_acc + prow0(pr) * kHeadDim) + d4;
  };
  for (int i = threadIdx.x; i < npairs * nslices; i += blockDim.x) {
    const int pr = i / nslices, sl = i % nslices;
    const int64_t p = prow0(pr) + sl;
    wts[i] = __ldcg(a.part_ml + p * 2);
    wts[npairs * nslices + i] = __ldcg(a.part_ml + p * 2 + 1);
  }
  __syncthreads();
  for (int pr = warp; pr < npairs; pr += nwarps)
    merge_weights_warp(wts + pr * nslices, wts + npairs * nslices + pr * nslices, nslices, lane);
  __syncthreads();
  for (int it = threadIdx.x; it < total; it += blockDim.x) {
    const int part = it % SPLIT, item = it / SPLIT;
    const int d4 = item % (kHeadDim / 4), pr = item / (kHeadDim / 4);
    const float* wm = wts + pr * nslices;
    const float4* src = acc_src(it);
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

}  // namespace ftkv
