// ftkv_device.cuh -- small device-side building blocks shared by the sm_103a kernels.
//
// E4M3FN conversions use the hardware packed converters (cvt ... e4m3x2): encode is
// round-to-nearest-even with .satfinite (out-of-range and +-Inf go to +-448, NaN to 0x7F), decode is
// exact (every E4M3FN value is an FP16 value).  Legacy warp-level tensor-core instructions (mma.sync,
// movmatrix) serve the small decode contractions; the prefill contraction uses tcgen05 (see
// prefill_tc.cu).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

namespace ftkv {

constexpr int kHeadDim = 128;
constexpr int kDevErrBadSlot = 0x1;
constexpr int kDevErrSeqLen = 0x2;
constexpr int kDevErrQRows = 0x4;
constexpr int kDevErrTimeout = 0x8;

// ---------------------------------------------------------------------------------------------
// E4M3FN codec
// ---------------------------------------------------------------------------------------------
// Two FP32 values -> two E4M3FN codes; `lo` lands in bits 0..7, `hi` in bits 8..15.
__device__ __forceinline__ uint32_t e4m3x2_encode(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3FN codes (bits 0..7 and 8..15) -> f16x2 with the same order (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t r;
  asm("{ .reg .b16 c; cvt.u16.u32 c, %1; cvt.rn.f16x2.e4m3x2 %0, c; }" : "=r"(r) : "r"(two_codes));
  return r;
}

// Low / high 16-bit halves of a 32-bit word of four codes -> f16x2.
__device__ __forceinline__ uint32_t e4m3_lo2(uint32_t w) { return e4m3x2_to_f16x2(w & 0xFFFFu); }
__device__ __forceinline__ uint32_t e4m3_hi2(uint32_t w) { return e4m3x2_to_f16x2(w >> 16); }

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t h) {
  __half2 v = *reinterpret_cast<__half2*>(&h);
  return __half22float2(v);
}

__device__ __forceinline__ uint32_t float2_to_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t float2_to_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Quantize-on-write of one 128-element BF16 row carried by a 16-lane half warp, lane l holding elements
// 8l .. 8l+7 in `raw` (FreeToken PR #853, "What changes": each row gets its own FP32 scale).  Row
// absmax = NaN-ignoring fmaxf from +0, scale = absmax / 448 (IEEE FP32 division), code =
// E4M3FN_rne_satfinite(x / scale) (the IEEE quotient, reached by Markstein's theorem below); an all-zero row
// keeps scale 0 and divides by 1.
// Every lane of the warp calls it: the max reduction shuffles within each 16-lane half.  Returns the
// lane's 8 codes (element 8l in the lowest byte) and sets `scale`.  The store kernel and the decode
// kernel's fused store both use this one definition.
template <int LANES = 16>  // lanes that carry one row (8 elements each): 16 for 128-d rows, 32 for 256-d
__device__ __forceinline__ uint2 quantize_row_lane8(const uint4 raw, float& scale) {
  float x[8];
  x[0] = bf16_lo(raw.x); x[1] = bf16_hi(raw.x);
  x[2] = bf16_lo(raw.y); x[3] = bf16_hi(raw.y);
  x[4] = bf16_lo(raw.z); x[5] = bf16_hi(raw.z);
  x[6] = bf16_lo(raw.w); x[7] = bf16_hi(raw.w);
  float amax = 0.0f;
  bool nan = false;
#pragma unroll
  for (int i = 0; i < 8; i++) {
    amax = fmaxf(amax, fabsf(x[i]));
    nan |= x[i] != x[i];
  }
#pragma unroll
  for (int off = 1; off < LANES; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  scale = __fdiv_rn(amax, 448.0f);
  const float div = (scale == 0.0f) ? 1.0f : scale;
  // The IEEE quotients x / div by Markstein's division theorem (P. Markstein, "Computation of elementary
  // functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with r = RN(1/div) and
  // q0 = RN(x r) (within an ulp of x / div), the remainder e = x - q0 div is exact in one FMA, and
  // RN(q0 + e r) is the correctly rounded x / div, provided nothing overflows or underflows.  Here
  // |x / div| <= 448 (no overflow).  A quotient that underflows FP32 is below 2^-126, far under half the
  // smallest E4M3 subnormal (2^-10), so its code is a signed zero either way.  A row whose div or 1/div is not
  // a normal number, or that holds a NaN, takes the IEEE division element by element.  (For x = -0 the steps
  // give +0; a quotient here has the sign of x, so the sign is copied from x.)
  const uint32_t de = (__float_as_uint(div) >> 23) & 0xFFu;
  float q[8];
  if (de >= 2u && de <= 252u && !nan) {
    const float r = __frcp_rn(div);
#pragma unroll
    for (int i = 0; i < 8; i++) {
      const float q0 = __fmul_rn(x[i], r);
      const float e = __fmaf_rn(-q0, div, x[i]);
      q[i] = copysignf(__fmaf_rn(e, r, q0), x[i]);  // the steps turn x = -0 into +0; the sign is x's anyway
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; i++) q[i] = __fdiv_rn(x[i], div);
  }
  const uint32_t w0 = e4m3x2_encode(q[0], q[1]), w1 = e4m3x2_encode(q[2], q[3]);
  const uint32_t w2 = e4m3x2_encode(q[4], q[5]), w3 = e4m3x2_encode(q[6], q[7]);
  return make_uint2(w0 | (w1 << 16), w2 | (w3 << 16));
}

// ---------------------------------------------------------------------------------------------
// Byte permute
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// ---------------------------------------------------------------------------------------------
// Warp-level tensor-core operations
// ---------------------------------------------------------------------------------------------
// D += A(16x16, f16, row) * B(16x8, f16, col), FP32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose an 8x8 matrix of 16-bit elements held in the standard fragment layout
// (lane i holds row i/4, columns 2*(i%4) and 2*(i%4)+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(a));
  return r;
}

// ---------------------------------------------------------------------------------------------
// Async copies global -> shared (Ampere-style cp.async, per thread)
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// L2 cache policy for data read once: its lines are the first to be evicted.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void cp_async_16_hint(uint32_t dst, const void* src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(pol) : "memory");
}

__device__ __forceinline__ void cp_async_4_hint(uint32_t dst, const void* src, uint64_t pol) {
  asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "l"(pol) : "memory");
}

// Bring the line holding p into L2 and keep it there in preference to other lines (a hint: no register, no
// ordering, no effect on correctness).
__device__ __forceinline__ void prefetch_l2_keep(const void* p) {
  asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p));
}

// Bulk L2 prefetch of [p, p + bytes): p 16-byte aligned, bytes a multiple of 16 (a hint, handled by the TMA unit).
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void st_shared_zero16(uint32_t dst) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0) : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t dst, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ void st_shared_u32(uint32_t dst, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(dst), "r"(v) : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

// Streaming 16-byte global load (read once; do not keep in L1).
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}

// Programmatic dependent launch.  Every kernel of this library is launched with programmatic stream
// serialization: the next kernel in the stream may be scheduled onto SMs this one has released while it
// drains.  Each kernel first allows its dependents to launch, then waits for its predecessor's completion
// and memory before touching global memory, so every result keeps plain stream order.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void flag_error(int* err, int bits) {
  if (err) atomicOr(err, bits);
}

}  // namespace ftkv
