// kv_rows.cu -- the FP8 row format's write and read kernels: quantize-on-write, reconstruction into
// the BF16 workspace, and the bare E4M3FN codec.
//
// Row format (FreeToken PR #853, "What changes"; issue #280, "Proof of concept"): one row = one
// token x one KV head = 128 E4M3FN codes + one FP32 scale.  scale = absmax / 448 (IEEE FP32
// division), code = E4M3FN_rne_satfinite(x / scale) (IEEE FP32 division); a row of zeros keeps scale
// 0 and divides by 1.  Both kernels are pure HBM streams; a warp moves whole rows with 16-byte
// accesses so every request is a full 32-byte sector run.
#include "ftkv_device.cuh"
#include "ftkv_internal.h"

namespace ftkv {

// ---------------------------------------------------------------------------------------------
// Quantize-on-write: one warp per (token, KV head).  Lanes 0..15 carry the K row, 16..31 the V row,
// 8 BF16 elements each.  Per row: NaN-ignoring absmax (fmaxf from +0), a 16-lane max reduction,
// one division for the scale, one division per element, packed saturating RNE encode.
// Bytes per (token, head): 2 x 256 B read, 2 x (128 B + 4 B) written, + the slot.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) store_quant_kernel(StoreArgs a) {
  const int64_t unit = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (unit >= a.num_tokens * a.num_kv_heads) return;
  const int lane = threadIdx.x & 31;
  const int64_t t = unit / a.num_kv_heads;
  const int h = static_cast<int>(unit % a.num_kv_heads);
  const int half = lane >> 4;   // 0: K, 1: V
  const int l = lane & 15;      // 8 elements per lane

  const int32_t slot = a.slots[t];
  if (slot < 0 || slot >= a.num_rows) {
    if (lane == 0) flag_error(a.err, kDevErrBadSlot);
    return;
  }
  const uint16_t* src = (half ? a.v : a.k) + (t * a.num_kv_heads + h) * kHeadDim + l * 8;
  const uint4 raw = ldg_stream16(src);
  float x[8];
  x[0] = bf16_lo(raw.x); x[1] = bf16_hi(raw.x);
  x[2] = bf16_lo(raw.y); x[3] = bf16_hi(raw.y);
  x[4] = bf16_lo(raw.z); x[5] = bf16_hi(raw.z);
  x[6] = bf16_lo(raw.w); x[7] = bf16_hi(raw.w);

  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; i++) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int off = 1; off < 16; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));

  const float scale = __fdiv_rn(amax, 448.0f);
  const float div = (scale == 0.0f) ? 1.0f : scale;
  uint32_t w0 = e4m3x2_encode(__fdiv_rn(x[0], div), __fdiv_rn(x[1], div));
  uint32_t w1 = e4m3x2_encode(__fdiv_rn(x[2], div), __fdiv_rn(x[3], div));
  uint32_t w2 = e4m3x2_encode(__fdiv_rn(x[4], div), __fdiv_rn(x[5], div));
  uint32_t w3 = e4m3x2_encode(__fdiv_rn(x[6], div), __fdiv_rn(x[7], div));
  uint2 packed = make_uint2(w0 | (w1 << 16), w2 | (w3 << 16));

  const int64_t row = static_cast<int64_t>(slot) * a.num_kv_heads + h;
  uint8_t* dst = (half ? a.v_codes : a.k_codes) + row * kHeadDim + l * 8;
  __stcs(reinterpret_cast<uint2*>(dst), packed);
  if (l == 0) __stcs((half ? a.v_scales : a.k_scales) + row, scale);
}

// ---------------------------------------------------------------------------------------------
// Reconstruct: 8 lanes per (logical row i, KV head h), 16 codes per lane for K and for V.
//   ws[i][h][d] = bf16_rne(float(decode(code)) * scale)   -- one FP32 product, no FMA contraction.
// Bytes per (row, head): 2 x (128 B + 4 B) read (scattered rows), 2 x 256 B written (dense).
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) reconstruct_kernel(ReconstructArgs a) {
  const int64_t unit = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3;
  if (unit >= a.num_prefix * a.num_kv_heads) return;
  const int l = threadIdx.x & 7;
  const int64_t i = unit / a.num_kv_heads;
  const int h = static_cast<int>(unit % a.num_kv_heads);
  int32_t slot = a.slots[i];
  if (slot < 0 || slot >= a.num_rows) {
    if (l == 0) flag_error(a.err, kDevErrBadSlot);
    slot = -1;
  }
  const int64_t dst_off = (i * a.num_kv_heads + h) * kHeadDim + l * 16;
  if (slot < 0) {  // skipped row: write zeros so the workspace holds no stale data
    uint4 z = make_uint4(0, 0, 0, 0);
    uint4* dk = reinterpret_cast<uint4*>(a.ws_k + dst_off);
    uint4* dv = reinterpret_cast<uint4*>(a.ws_v + dst_off);
    dk[0] = z; dk[1] = z; dv[0] = z; dv[1] = z;
    return;
  }
  const int64_t row = static_cast<int64_t>(slot) * a.num_kv_heads + h;
  const uint4 kc = ldg_stream16(a.k_codes + row * kHeadDim + l * 16);
  const uint4 vc = ldg_stream16(a.v_codes + row * kHeadDim + l * 16);
  const float ks = __ldg(a.k_scales + row);
  const float vs = __ldg(a.v_scales + row);

  auto expand = [](const uint4& c, float s, uint4& o0, uint4& o1) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    uint32_t out[8];
#pragma unroll
    for (int j = 0; j < 4; j++) {
      float2 lo = f16x2_to_float2(e4m3_lo2(w[j]));
      float2 hi = f16x2_to_float2(e4m3_hi2(w[j]));
      out[2 * j] = float2_to_bf16x2(__fmul_rn(lo.x, s), __fmul_rn(lo.y, s));
      out[2 * j + 1] = float2_to_bf16x2(__fmul_rn(hi.x, s), __fmul_rn(hi.y, s));
    }
    o0 = make_uint4(out[0], out[1], out[2], out[3]);
    o1 = make_uint4(out[4], out[5], out[6], out[7]);
  };
  uint4 k0, k1, v0, v1;
  expand(kc, ks, k0, k1);
  expand(vc, vs, v0, v1);
  uint4* dk = reinterpret_cast<uint4*>(a.ws_k + dst_off);
  uint4* dv = reinterpret_cast<uint4*>(a.ws_v + dst_off);
  dk[0] = k0; dk[1] = k1;
  dv[0] = v0; dv[1] = v1;
}

// ---------------------------------------------------------------------------------------------
// Bare codec (same device conversions as above), one element per thread, no alignment needed.
// ---------------------------------------------------------------------------------------------
__global__ void e4m3_encode_kernel(const float* __restrict__ x, uint8_t* __restrict__ c, int64_t n) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    c[i] = static_cast<uint8_t>(e4m3x2_encode(x[i], 0.0f) & 0xFFu);
}

__global__ void e4m3_decode_kernel(const uint8_t* __restrict__ c, float* __restrict__ x, int64_t n) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    x[i] = f16x2_to_float2(e4m3x2_to_f16x2(c[i])).x;
}

// ---------------------------------------------------------------------------------------------
cudaError_t launch_store_quant(const StoreArgs& a, cudaStream_t s) {
  const int64_t warps = a.num_tokens * a.num_kv_heads;
  const int64_t blocks = (warps * 32 + 255) / 256;
  store_quant_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_reconstruct(const ReconstructArgs& a, cudaStream_t s) {
  const int64_t units = a.num_prefix * a.num_kv_heads;
  const int64_t blocks = (units * 8 + 255) / 256;
  reconstruct_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_e4m3_encode(const float* x, uint8_t* c, int64_t n, int num_sms, cudaStream_t s) {
  int64_t blocks = (n + 255) / 256;
  if (blocks > static_cast<int64_t>(num_sms) * 32) blocks = static_cast<int64_t>(num_sms) * 32;
  e4m3_encode_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(x, c, n);
  return cudaGetLastError();
}

cudaError_t launch_e4m3_decode(const uint8_t* c, float* x, int64_t n, int num_sms, cudaStream_t s) {
  int64_t blocks = (n + 255) / 256;
  if (blocks > static_cast<int64_t>(num_sms) * 32) blocks = static_cast<int64_t>(num_sms) * 32;
  e4m3_decode_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(c, x, n);
  return cudaGetLastError();
}

}  // namespace ftkv
