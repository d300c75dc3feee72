// kv_rows.cu -- the FP8 row format's write and read kernels: quantize-on-write, reconstruction into
// the BF16 workspace, and the bare E4M3FN codec.
//
// Row format (FreeToken PR #853, "What changes"; issue #280, "Proof of concept"): one row = one
// token x one KV head = head_dim (128, or 256 for the store and the single-row decode) E4M3FN codes + one
// FP32 scale.  scale = absmax / 448 (IEEE FP32
// division), code = E4M3FN_rne_satfinite(x / scale) (IEEE FP32 division); a row of zeros keeps scale
// 0 and divides by 1.  Both kernels are pure HBM streams; a warp moves whole rows with 16-byte
// accesses so every request is a full 32-byte sector run.
#include "ftkv_device.cuh"
#include "ftkv_internal.h"

namespace ftkv {

// ---------------------------------------------------------------------------------------------
// Quantize-on-write.  Half a warp carries one 128-d row (token, KV head, tensor): 16 lanes x 8 BF16
// elements; a 256-d row takes a whole warp (32 lanes x 8), and a (token, head) pair two warps (K, V).
// A warp handles STORE_UNITS (token, head) pairs -- K and V rows of each -- and issues all its loads
// before any arithmetic.  One pair per warp: more warps in flight hide the arithmetic's latency better
// than longer load batches per warp (48-layer store: 1 pair 431 us, 2 pairs 468 us, 4 pairs 618 us).
// Per row: NaN-ignoring absmax (fmaxf from +0), a 16-lane max reduction, scale = absmax / 448 (IEEE
// division), then the IEEE quotient x / scale for every element, by one reciprocal per row and a product
// and two FMAs per element (Markstein's theorem; rows whose scale or its reciprocal is not a normal number,
// or that hold a NaN, divide element by element: quantize_row_lane8).
// Bytes per (token, head): 2 x 256 B read, 2 x (128 B + 4 B) written, + the slot.
// ---------------------------------------------------------------------------------------------
constexpr int STORE_UNITS = 1;  // the loop form is kept so the batch size stays a one-line choice

// (unit / hkv, unit % hkv) without a 64-bit integer division (a long software sequence): a shift for
// power-of-two head counts, a 32-bit division when the unit fits, the 64-bit one otherwise.
__device__ __forceinline__ void split_unit(int64_t unit, int hkv, int64_t& t, int& h) {
  if ((hkv & (hkv - 1)) == 0) {
    const int sh = __ffs(hkv) - 1;
    t = unit >> sh;
    h = static_cast<int>(unit & (hkv - 1));
  } else if (unit < 0x7FFFFFFF) {
    const uint32_t u = static_cast<uint32_t>(unit);
    t = u / static_cast<uint32_t>(hkv);
    h = static_cast<int>(u % static_cast<uint32_t>(hkv));
  } else {
    t = unit / hkv;
    h = static_cast<int>(unit % hkv);
  }
}

template <int D>
__global__ void __launch_bounds__(256) store_quant_kernel(StoreArgs a) {
  pdl_enter();
  constexpr int LPR = D / 8;    // lanes per row, 8 elements each
  const int64_t gwarp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  // D = 128: one warp per pair, K on lanes 0-15 and V on 16-31; D = 256: warp 2u carries K, 2u + 1 V
  const int64_t warp_id = (D == 128) ? gwarp : gwarp >> 1;
  const int half = (D == 128) ? lane >> 4 : static_cast<int>(gwarp & 1);  // 0: K, 1: V
  const int l = lane % LPR;
  const int64_t total = a.num_tokens * a.num_kv_heads;
  uint4 raw[STORE_UNITS];
  int32_t slot[STORE_UNITS];
#pragma unroll
  for (int u = 0; u < STORE_UNITS; u++) {
    const int64_t unit = warp_id * STORE_UNITS + u;
    slot[u] = -1;
    raw[u] = make_uint4(0, 0, 0, 0);
    if (unit < total) {
      int64_t t;
      int h;
      split_unit(unit, a.num_kv_heads, t, h);
      slot[u] = __ldg(a.slots + t);
      raw[u] = ldg_stream16((half ? a.v : a.k) + (t * a.num_kv_heads + h) * D + l * 8);
    }
  }
#pragma unroll
  for (int u = 0; u < STORE_UNITS; u++) {
    const int64_t unit = warp_id * STORE_UNITS + u;
    if (unit >= total) break;  // warp-uniform
    int64_t t;
    int h;
    split_unit(unit, a.num_kv_heads, t, h);
    float scale;
    const uint2 packed = quantize_row_lane8<LPR>(raw[u], scale);  // every lane: the reduction shuffles
    if (slot[u] < 0 || slot[u] >= a.num_rows) {
      if (lane == 0) flag_error(a.err, kDevErrBadSlot);
      continue;
    }
    const int64_t row = static_cast<int64_t>(slot[u]) * a.num_kv_heads + h;
    __stcs(reinterpret_cast<uint2*>((half ? a.v_codes : a.k_codes) + row * D + l * 8), packed);
    if (l == 0) __stcs((half ? a.v_scales : a.k_scales) + row, scale);
  }
}

// ---------------------------------------------------------------------------------------------
// Reconstruct: 8 lanes per (logical row i, KV head h), 16 codes per lane for K and for V; each lane
// handles RECON_UNITS such units with every load issued before any conversion.  One unit per lane: the
// scattered code rows are latency-bound, and more warps in flight beat longer batches (8 launches over
// 14,336 rows: 1 unit 51.0 us, 2 units 61.0 us, 4 units 66.3 us).
//   ws[i][h][d] = bf16_rne(float(decode(code)) * scale)   -- one FP32 product, no FMA contraction.
// Bytes per (row, head): 2 x (128 B + 4 B) read (scattered rows), 2 x 256 B written (dense).
// ---------------------------------------------------------------------------------------------
constexpr int RECON_UNITS = 1;

__device__ __forceinline__ void expand16(const uint4& c, float s, uint4& o0, uint4& o1) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  uint32_t out[8];
#pragma unroll
  for (int j = 0; j < 4; j++) {
    const float2 lo = f16x2_to_float2(e4m3_lo2(w[j]));
    const float2 hi = f16x2_to_float2(e4m3_hi2(w[j]));
    out[2 * j] = float2_to_bf16x2(__fmul_rn(lo.x, s), __fmul_rn(lo.y, s));
    out[2 * j + 1] = float2_to_bf16x2(__fmul_rn(hi.x, s), __fmul_rn(hi.y, s));
  }
  o0 = make_uint4(out[0], out[1], out[2], out[3]);
  o1 = make_uint4(out[4], out[5], out[6], out[7]);
}

__global__ void __launch_bounds__(256) reconstruct_kernel(ReconstructArgs a) {
  pdl_enter();
  const int64_t group = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3;
  const int l = threadIdx.x & 7;
  const int64_t total = a.num_prefix * a.num_kv_heads;
  int32_t slot[RECON_UNITS];
#pragma unroll
  for (int u = 0; u < RECON_UNITS; u++) {
    const int64_t unit = group * RECON_UNITS + u;
    int64_t t;
    int h;
    split_unit(unit, a.num_kv_heads, t, h);
    slot[u] = (unit < total) ? __ldg(a.slots + t) : -1;
  }
  uint4 kc[RECON_UNITS], vc[RECON_UNITS];
  float ks[RECON_UNITS], vs[RECON_UNITS];
#pragma unroll
  for (int u = 0; u < RECON_UNITS; u++) {
    const int64_t unit = group * RECON_UNITS + u;
    int64_t t;
    int h;
    split_unit(unit, a.num_kv_heads, t, h);
    const bool ok = unit < total && slot[u] >= 0 && slot[u] < a.num_rows;
    const int64_t row = ok ? static_cast<int64_t>(slot[u]) * a.num_kv_heads + h : 0;
    kc[u] = ok ? ldg_stream16(a.k_codes + row * kHeadDim + l * 16) : make_uint4(0, 0, 0, 0);
    vc[u] = ok ? ldg_stream16(a.v_codes + row * kHeadDim + l * 16) : make_uint4(0, 0, 0, 0);
    ks[u] = ok ? __ldg(a.k_scales + row) : 0.0f;
    vs[u] = ok ? __ldg(a.v_scales + row) : 0.0f;
  }
#pragma unroll
  for (int u = 0; u < RECON_UNITS; u++) {
    const int64_t unit = group * RECON_UNITS + u;
    if (unit >= total) break;
    if ((slot[u] < 0 || slot[u] >= a.num_rows) && l == 0) flag_error(a.err, kDevErrBadSlot);
    // a skipped row is written as zeros so the workspace holds no stale data
    uint4 k0, k1, v0, v1;
    expand16(kc[u], ks[u], k0, k1);
    expand16(vc[u], vs[u], v0, v1);
    const int64_t dst_off = unit * kHeadDim + l * 16;   // unit = i * Hkv + h
    uint4* dk = reinterpret_cast<uint4*>(a.ws_k + dst_off);
    uint4* dv = reinterpret_cast<uint4*>(a.ws_v + dst_off);
    dk[0] = k0; dk[1] = k1;
    dv[0] = v0; dv[1] = v1;
  }
}

// ---------------------------------------------------------------------------------------------
// Bare codec (same device conversions as above), one element per thread, no alignment needed.
// ---------------------------------------------------------------------------------------------
__global__ void e4m3_encode_kernel(const float* __restrict__ x, uint8_t* __restrict__ c, int64_t n) {
  pdl_enter();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    c[i] = static_cast<uint8_t>(e4m3x2_encode(x[i], 0.0f) & 0xFFu);
}

__global__ void e4m3_decode_kernel(const uint8_t* __restrict__ c, float* __restrict__ x, int64_t n) {
  pdl_enter();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    x[i] = f16x2_to_float2(e4m3x2_to_f16x2(c[i])).x;
}

// ---------------------------------------------------------------------------------------------
cudaError_t launch_store_quant(const StoreArgs& a, cudaStream_t s) {
  const int64_t warps = (a.num_tokens * a.num_kv_heads + STORE_UNITS - 1) / STORE_UNITS * (a.head_dim / 128);
  const int64_t blocks = (warps * 32 + 255) / 256;
  if (a.head_dim == 256)
    return launch_k(store_quant_kernel<256>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, a);
  return launch_k(store_quant_kernel<128>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, a);
}

cudaError_t launch_reconstruct(const ReconstructArgs& a, cudaStream_t s) {
  const int64_t groups = (a.num_prefix * a.num_kv_heads + RECON_UNITS - 1) / RECON_UNITS;
  const int64_t blocks = (groups * 8 + 255) / 256;
  return launch_k(reconstruct_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, a);
}

cudaError_t launch_e4m3_encode(const float* x, uint8_t* c, int64_t n, int num_sms, cudaStream_t s) {
  int64_t blocks = (n + 255) / 256;
  if (blocks > static_cast<int64_t>(num_sms) * 32) blocks = static_cast<int64_t>(num_sms) * 32;
  return launch_k(e4m3_encode_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, x, c, n);
}

cudaError_t launch_e4m3_decode(const uint8_t* c, float* x, int64_t n, int num_sms, cudaStream_t s) {
  int64_t blocks = (n + 255) / 256;
  if (blocks > static_cast<int64_t>(num_sms) * 32) blocks = static_cast<int64_t>(num_sms) * 32;
  return launch_k(e4m3_decode_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, c, x, n);
}

}  // namespace ftkv
