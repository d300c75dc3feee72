// prefill_mma.cu -- prefill (extend) attention on the legacy warp-level tensor-core path.
//
// What it computes (FreeToken PR #853, "What changes"): chunk query t attends to every key of the
// reconstructed BF16 prefix and to chunk keys 0..t; K/V of the current chunk stay BF16.
// This kernel is the mma.sync (m16n8k16, BF16 in, FP32 accumulate) formulation: 64 query rows of
// one head per CTA (16 per warp), 64-key tiles double-buffered through shared memory with cp.async,
// FA2-style online softmax in registers.  The tcgen05 kernel (prefill_tc.cu) is the fast path; this
// one is kept as a comparison point and as an independent second implementation on the GPU.
#include "ftkv_device.cuh"
#include "ftkv_internal.h"

namespace ftkv {
namespace {

constexpr int BM = 64;   // query rows per CTA
constexpr int BN = 64;   // keys per tile
constexpr int ROWB = kHeadDim * 2;  // 256 bytes per BF16 row
constexpr int TILE_BYTES = BN * ROWB;  // 16 KB
constexpr int SMEM = BM * ROWB + 2 * 2 * TILE_BYTES;  // Q + 2 stages x (K, V) = 80 KB

// 16-byte chunk c (0..15) of row r of a [rows][256 B] tile, XOR-swizzled on the low 3 bits.
__device__ __forceinline__ uint32_t sw(int r, int c) { return r * ROWB + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void cp_async_16_zfill(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}

// Copy rows [r0, r0+BN) of a [rows][heads][128] BF16 tensor (head hk) into a swizzled tile;
// rows >= nrows are zero-filled.
__device__ __forceinline__ void load_tile(uint32_t dst, const uint16_t* base, int64_t nrows, int heads,
                                          int hk, int64_t r0) {
  for (int i = threadIdx.x; i < BN * 16; i += blockDim.x) {
    const int r = i >> 4, c = i & 15;
    const int64_t gr = r0 + r;
    const bool valid = gr < nrows;
    const uint16_t* src = valid ? base + (gr * heads + hk) * kHeadDim + c * 8 : base;
    cp_async_16_zfill(dst + sw(r, c), src, valid);
  }
}

__global__ void __launch_bounds__(128) prefill_mma_kernel(const PrefillArgs a) {
  pdl_enter();
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = smem_addr(smem);
  const uint32_t sKV = sQ + BM * ROWB;  // stage s: K at sKV + s*2*TILE, V at + TILE
  const int hq = blockIdx.y;
  const int hk = hq / (a.num_q_heads / a.num_kv_heads);
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * BM;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;

  // Q tile (zero-filled past the chunk)
  for (int i = threadIdx.x; i < BM * 16; i += blockDim.x) {
    const int r = i >> 4, c = i & 15;
    const int64_t gr = t0 + r;
    const bool valid = gr < a.chunk_len;
    const uint16_t* src = valid ? a.q + (gr * a.num_q_heads + hq) * kHeadDim + c * 8 : a.q;
    cp_async_16_zfill(sQ + sw(r, c), src, valid);
  }
  cp_async_commit();

  const int64_t n_prefix_tiles = (a.prefix_len + BN - 1) / BN;
  int64_t last_q = t0 + BM - 1;
  if (last_q > a.chunk_len - 1) last_q = a.chunk_len - 1;
  const int64_t n_chunk_tiles = last_q / BN + 1;
  const int64_t n_tiles = n_prefix_tiles + n_chunk_tiles;

  auto issue = [&](int64_t kt, int stage) {
    const uint32_t dK = sKV + stage * 2 * TILE_BYTES, dV = dK + TILE_BYTES;
    if (kt < n_prefix_tiles) {
      load_tile(dK, a.ws_k, a.prefix_len, a.num_kv_heads, hk, kt * BN);
      load_tile(dV, a.ws_v, a.prefix_len, a.num_kv_heads, hk, kt * BN);
    } else {
      const int64_t r0 = (kt - n_prefix_tiles) * BN;
      load_tile(dK, a.k_chunk, a.chunk_len, a.num_kv_heads, hk, r0);
      load_tile(dV, a.v_chunk, a.chunk_len, a.num_kv_heads, hk, r0);
    }
    cp_async_commit();
  };
  issue(0, 0);
  cp_async_wait<1>();  // Q landed
  __syncthreads();

  // Q fragments (A operand): rows warp*16 + {g, g+8}, 8 k-steps
  uint32_t qa[8][4];
#pragma unroll
  for (int kk = 0; kk < 8; kk++) {
    const int r = warp * 16 + (lane & 15);
    const int c = 2 * kk + (lane >> 4);
    ldsm_x4(sQ + sw(r, c), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
  }

  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; i++) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.0f, 0.0f};
  const int64_t qrow[2] = {t0 + warp * 16 + g, t0 + warp * 16 + g + 8};

  for (int64_t kt = 0; kt < n_tiles; kt++) {
    const int stage = static_cast<int>(kt & 1);
    if (kt + 1 < n_tiles) issue(kt + 1, stage ^ 1); else cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint32_t sK = sKV + stage * 2 * TILE_BYTES, sV = sK + TILE_BYTES;

    // S = Q K^T : 16 rows x 64 keys per warp
    float sc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; nt++) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.0f;
#pragma unroll
    for (int kk = 0; kk < 8; kk++) {
#pragma unroll
      for (int np = 0; np < 4; np++) {
        uint32_t b0, b1, b2, b3;
        const int key = np * 16 + ((lane >> 4) << 3) + (lane & 7);
        const int c = 2 * kk + ((lane >> 3) & 1);
        ldsm_x4(sK + sw(key, c), b0, b1, b2, b3);
        mma_bf16_16816(sc[2 * np], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
        mma_bf16_16816(sc[2 * np + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
      }
    }
    // scale + mask: key index of column (nt, e) is base + nt*8 + 2t + e
    const bool is_prefix = kt < n_prefix_tiles;
    const int64_t kbase = is_prefix ? kt * BN : (kt - n_prefix_tiles) * BN;
    float bm[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; nt++)
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const int64_t key = kbase + nt * 8 + 2 * t + (e & 1);
        const int rr = e >> 1;
        bool ok;
        if (is_prefix) ok = key < a.prefix_len;
        else ok = key <= qrow[rr] && key < a.chunk_len;
        const float v = ok ? sc[nt][e] * a.qk_scale_log2 : -INFINITY;
        sc[nt][e] = v;
        bm[rr] = fmaxf(bm[rr], v);
      }
    float alpha[2], mu[2];
#pragma unroll
    for (int rr = 0; rr < 2; rr++) {
      bm[rr] = fmaxf(bm[rr], __shfl_xor_sync(0xffffffffu, bm[rr], 1));
      bm[rr] = fmaxf(bm[rr], __shfl_xor_sync(0xffffffffu, bm[rr], 2));
      const float mn = fmaxf(mrow[rr], bm[rr]);
      mu[rr] = (mn == -INFINITY) ? 0.0f : mn;
      alpha[rr] = exp2f(mrow[rr] - mu[rr]);
      mrow[rr] = mn;
    }
    float ps[2] = {0.0f, 0.0f};
    uint32_t pa[4][4];
#pragma unroll
    for (int nt = 0; nt < 8; nt++) {
      const float p0 = exp2f(sc[nt][0] - mu[0]), p1 = exp2f(sc[nt][1] - mu[0]);
      const float p2 = exp2f(sc[nt][2] - mu[1]), p3 = exp2f(sc[nt][3] - mu[1]);
      ps[0] += p0 + p1;
      ps[1] += p2 + p3;
      const int kk = nt >> 1, hi = nt & 1;
      pa[kk][hi ? 2 : 0] = float2_to_bf16x2(p0, p1);
      pa[kk][hi ? 3 : 1] = float2_to_bf16x2(p2, p3);
    }
    lrow[0] = lrow[0] * alpha[0] + ps[0];
    lrow[1] = lrow[1] * alpha[1] + ps[1];
#pragma unroll
    for (int i = 0; i < 16; i++) {
      o[i][0] *= alpha[0];
      o[i][1] *= alpha[0];
      o[i][2] *= alpha[1];
      o[i][3] *= alpha[1];
    }
    // O += P V : 16 rows x 128 d
#pragma unroll
    for (int kk = 0; kk < 4; kk++) {
#pragma unroll
      for (int dp = 0; dp < 8; dp++) {
        uint32_t b0, b1, b2, b3;
        const int key = kk * 16 + (lane & 15);
        const int c = 2 * dp + (lane >> 4);
        ldsm_x4_t(sV + sw(key, c), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * dp], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
        mma_bf16_16816(o[2 * dp + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
      }
    }
    __syncthreads();  // stage free for the next issue
  }
  cp_async_wait<0>();

#pragma unroll
  for (int rr = 0; rr < 2; rr++) {
    lrow[rr] += __shfl_xor_sync(0xffffffffu, lrow[rr], 1);
    lrow[rr] += __shfl_xor_sync(0xffffffffu, lrow[rr], 2);
  }
#pragma unroll
  for (int rr = 0; rr < 2; rr++) {
    if (qrow[rr] >= a.chunk_len) continue;
    const float inv = lrow[rr] > 0.0f ? 1.0f / lrow[rr] : 0.0f;
    uint32_t* dst = reinterpret_cast<uint32_t*>(a.out + (qrow[rr] * a.num_q_heads + hq) * kHeadDim);
#pragma unroll
    for (int i = 0; i < 16; i++) dst[i * 4 + t] = float2_to_bf16x2(o[i][2 * rr] * inv, o[i][2 * rr + 1] * inv);
  }
}

}  // namespace

cudaError_t launch_prefill_mma(const PrefillArgs& a, cudaStream_t s) {
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(prefill_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  dim3 grid(static_cast<unsigned>((a.chunk_len + BM - 1) / BM), a.num_q_heads);
  return launch_k(prefill_mma_kernel, grid, dim3(128), SMEM, s, a);
}

}  // namespace ftkv
