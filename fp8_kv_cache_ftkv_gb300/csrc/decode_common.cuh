// decode_common.cuh -- pieces shared by the split-K decode kernels (decode_mr.cu: one KV head per CTA,
// multi-row batches; decode_tok.cu: every KV head of a token per CTA, single-row batches; bf16_pool.cu:
// the same over a BF16 pool).
//
// The split merge after a grid barrier (cooperative launches) lives here as well:
// for each (query row, query head), with per-slice maximum m_s (log2 units), sum l_s and unnormalized
// accumulator O_s (FreeToken PR #897, "Fresh R9700 stage-1 A/B": a stage over key slices, then a merge)
//     M = max_s m_s,   L = sum_s 2^(m_s - M) l_s,   o = sum_s (2^(m_s - M) / L) O_s      (o = 0 if L = 0).
#pragma once

#include <cfloat>

#include "ftkv_device.cuh"
#include "ftkv_internal.h"

namespace ftkv {

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// D += A(16x32, e4m3, row) * B(32x8, e4m3, col), FP32 accumulate.
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ int64_t clamp_seq_len(const DecodeArgs& a, int b, bool report) {
  int64_t n = a.seq_lens[b];
  const int64_t nmax = a.max_seq_len < a.req_stride ? a.max_seq_len : a.req_stride;
  if (n < 0 || n > nmax) {
    if (report) flag_error(a.err, kDevErrSeqLen);
    n = n < 0 ? 0 : nmax;
  }
  return n;
}

// First key of a request's attended range: 0, or with a sliding window of W keys the window start of its first
// query row (row 0 of R sees keys 0 .. n-R, so its window starts at n-R+1-W).  The key slices of a request
// cover keys [first, n).
__device__ __forceinline__ int64_t first_key(const DecodeArgs& a, int64_t n, int R) {
  if (a.window <= 0) return 0;
  const int64_t lo = n - R + 1 - a.window;
  return lo > 0 ? lo : 0;
}

// Wait for the preceding grid of the stream (programmatic dependent launch) -- its completion and memory.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Barrier of key group gi (named barrier 1 + gi, immediate ids so that only NG + 1 barriers are used).
template <int NG>
__device__ __forceinline__ void group_barrier(int gi, int count) {
  if (NG == 1 || gi == 0) { asm volatile("bar.sync 1, %0;" ::"r"(count) : "memory"); return; }
  if (NG == 2 || gi == 1) { asm volatile("bar.sync 2, %0;" ::"r"(count) : "memory"); return; }
  if (NG == 4) {
    if (gi == 2) asm volatile("bar.sync 3, %0;" ::"r"(count) : "memory");
    else asm volatile("bar.sync 4, %0;" ::"r"(count) : "memory");
    return;
  }
  switch (gi) {
    case 2: asm volatile("bar.sync 3, %0;" ::"r"(count) : "memory"); break;
    case 3: asm volatile("bar.sync 4, %0;" ::"r"(count) : "memory"); break;
    case 4: asm volatile("bar.sync 5, %0;" ::"r"(count) : "memory"); break;
    case 5: asm volatile("bar.sync 6, %0;" ::"r"(count) : "memory"); break;
    case 6: asm volatile("bar.sync 7, %0;" ::"r"(count) : "memory"); break;
    default: asm volatile("bar.sync 8, %0;" ::"r"(count) : "memory"); break;
  }
}

__device__ __forceinline__ float exp2i(int e) {  // 2^e for -126 <= e <= 127, exact
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// ---- merge of one output item: (query row t, query head qh, 4 of the 128 d), by one warp ----
// Lane k takes the partials k, k + 32, ... of the (row, head) in rounds of 32 * CH (one round in the usual
// case): their (m, l) and their 4 accumulators, every load of a round in flight at once; the round maximum by
// a warp reduction, the lane's running (M, L, o) rescaled when it grows; L and o reduced across the lanes at
// the end.  Requests whose row offsets are inconsistent were skipped by the main kernel (flagged there) and
// are skipped here; a (row, head) without keys gets zeros.
template <int CH>
__device__ __forceinline__ void merge_item(const DecodeArgs& a, int64_t it, int lane) {
  const int QUADS = a.head_dim / 4;
  const int64_t t = it / (a.num_q_heads * QUADS);  // query row
  const int rem = static_cast<int>(it - t * a.num_q_heads * QUADS);
  const int qh = rem / QUADS, d4 = rem % QUADS;
  int b = static_cast<int>(t), R = 1;
  if (a.q_row_offsets) {  // request of row t
    int lo = 0, hi = a.batch;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (a.q_row_offsets[mid + 1] <= t) lo = mid + 1; else hi = mid;
    }
    b = lo;
    if (b >= a.batch) return;
    const int64_t r0 = a.q_row_offsets[b];
    R = a.q_row_offsets[b + 1] - a.q_row_offsets[b];
    if (R < 0 || R > a.max_q_rows || r0 < 0 || r0 + R > a.total_q_rows) return;  // skipped request
  }
  int64_t n = a.seq_lens[b];
  const int64_t nmax = a.max_seq_len < a.req_stride ? a.max_seq_len : a.req_stride;
  n = n < 0 ? 0 : (n > nmax ? nmax : n);
  const int64_t nsl64 = (n - first_key(a, n, R) + a.chunk - 1) / a.chunk;
  const int nslices = static_cast<int>(nsl64 < a.num_splits ? nsl64 : a.num_splits) * a.pps;
  uint16_t* dst = a.out + (t * a.num_q_heads + qh) * a.head_dim + 4 * d4;
  if (nslices == 0) {  // no keys: zeros
    if (lane == 0) *reinterpret_cast<uint2*>(dst) = make_uint2(0u, 0u);
    return;
  }
  const int64_t np = static_cast<int64_t>(a.num_splits) * a.pps;  // partial slots per (row, head)
  const int64_t prow0 = (t * a.num_q_heads + qh) * np;
  const float2* pml = reinterpret_cast<const float2*>(a.part_ml) + prow0;
  // slice sl's 4 accumulators: pacc[sl * pst]
  const float4* pacc = a.ptrans
                           ? reinterpret_cast<const float4*>(a.part_acc) + ((t * a.num_q_heads + qh) * QUADS + d4) * np
                           : reinterpret_cast<const float4*>(a.part_acc + prow0 * a.head_dim) + d4;
  const int pst = a.ptrans ? 1 : QUADS;
  float M = -INFINITY, L = 0.0f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int base = 0; base < nslices; base += 32 * CH) {  // warp-uniform
    float2 ml[CH];
    float4 v[CH];
#pragma unroll
    for (int k = 0; k < CH; k++) {
      const int sl = base + lane + 32 * k;
      const bool in = sl < nslices;
      ml[k] = in ? __ldcg(pml + sl) : make_float2(-INFINITY, 0.f);
      v[k] = in ? __ldcg(pacc + static_cast<int64_t>(sl) * pst) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float Mc = M;
#pragma unroll
    for (int k = 0; k < CH; k++) Mc = fmaxf(Mc, ml[k].x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) Mc = fmaxf(Mc, __shfl_xor_sync(0xffffffffu, Mc, off));
    if (Mc == -INFINITY) continue;  // warp-uniform: nothing seen yet
    const float sc = (M == -INFINITY) ? 0.0f : fast_exp2(M - Mc);
    L *= sc;
    o.x *= sc;
    o.y *= sc;
    o.z *= sc;
    o.w *= sc;
#pragma unroll
    for (int k = 0; k < CH; k++) {
      const float w = (ml[k].x == -INFINITY) ? 0.0f : fast_exp2(ml[k].x - Mc);
      L = fmaf(w, ml[k].y, L);
      o.x = fmaf(w, v[k].x, o.x);
      o.y = fmaf(w, v[k].y, o.y);
      o.z = fmaf(w, v[k].z, o.z);
      o.w = fmaf(w, v[k].w, o.w);
    }
    M = Mc;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    L += __shfl_xor_sync(0xffffffffu, L, off);
    o.x += __shfl_xor_sync(0xffffffffu, o.x, off);
    o.y += __shfl_xor_sync(0xffffffffu, o.y, off);
    o.z += __shfl_xor_sync(0xffffffffu, o.z, off);
    o.w += __shfl_xor_sync(0xffffffffu, o.w, off);
  }
  const float invL = (M != -INFINITY && L > 0.0f) ? 1.0f / L : 0.0f;
  if (lane == 0)
    *reinterpret_cast<uint2*>(dst) =
        make_uint2(float2_to_bf16x2(o.x * invL, o.y * invL), float2_to_bf16x2(o.z * invL, o.w * invL));
}

// ---- cooperative finish: the split merge after a grid barrier, spread over every warp of the grid ----
// Used when the whole grid is resident at once (cooperative launch).  Every CTA calls it exactly once,
// after publishing its partials (or instead of doing anything, if its slice holds no keys).
// The barrier needs no reset: gbar[0] counts the arrivals of every call on this workspace (it only grows, and
// wraps), and gbar[1] holds its value at the end of the previous call's barrier.  Each CTA reads gbar[1] = B
// before it arrives, so every CTA of a call reads the same B; the CTA whose arrival completes the call (ticket
// B + ncta - 1) stores B + ncta into gbar[1] for the next call, which reads it only after this kernel has
// completed.  Waiting is polled by thread 0, bounded at 2 s (a timeout is flagged and the merge skipped).
// Then output item (query row, query head, 4 of the 128 d) i goes to warp i / ncta of CTA i % ncta
// (merge_item).
template <int WARPS>
__device__ __forceinline__ void coop_finish(const DecodeArgs& a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ncta = gridDim.x * gridDim.y * gridDim.z;
  const int cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  __syncthreads();  // every thread's partials are written before thread 0 releases them
  __shared__ int s_ok;
  if (threadIdx.x == 0) {
    // unsigned arithmetic: the counters wrap
    const unsigned base = *reinterpret_cast<volatile unsigned*>(a.gbar + 1);
    const unsigned target = base + static_cast<unsigned>(ncta);
    unsigned ticket;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(ticket) : "l"(a.gbar) : "memory");
    if (ticket == target - 1u) a.gbar[1] = static_cast<int>(target);  // read by the next call only
    unsigned long long t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    unsigned v = ticket + 1u;
    bool ok = static_cast<int>(v - target) >= 0;
    while (!ok) {
      __nanosleep(32);
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a.gbar) : "memory");
      ok = static_cast<int>(v - target) >= 0;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (!ok && t - t0 > 2000000000ull) break;
    }
    if (!ok) flag_error(a.err, kDevErrTimeout);
    s_ok = ok;
  }
  __syncthreads();
  if (s_ok) {
    const int64_t items = a.total_q_rows * a.num_q_heads * (a.head_dim / 4);
    for (int64_t it = cta + static_cast<int64_t>(ncta) * warp; it < items; it += static_cast<int64_t>(ncta) * WARPS)
      merge_item<10>(a, it, lane);
  }
}

// ---- the split merge as a kernel of its own, launched right behind a split-K decode kernel whose grid does not
// fit on the GPU at once (no cooperative launch, hence no grid barrier).  One warp per output item (query row,
// query head, 4 of the 128 d); the grid waits for the decode kernel (programmatic dependent launch). ----
constexpr int kMergeWarps = 4;  // warps per merge CTA
template <int MW>
__global__ void __launch_bounds__(MW * 32) decode_merge_kernel(const DecodeArgs a) {
  griddep_launch_dependents();
  griddep_wait();
  const int64_t it = static_cast<int64_t>(blockIdx.x) * MW + (threadIdx.x >> 5);
  if (it < a.total_q_rows * a.num_q_heads * (a.head_dim / 4)) merge_item<10>(a, it, threadIdx.x & 31);
}

}  // namespace ftkv
