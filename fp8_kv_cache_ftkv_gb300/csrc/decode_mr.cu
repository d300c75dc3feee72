// decode_mr.cu -- split-K decode attention for multi-row requests on the sm_100-family tensor cores (tcgen05 +
// TMEM), computing what decode.cu defines (FreeToken PR #897, opening description and "Fresh R9700 stage-1
// A/B"; row r of a request's R rows sees keys 0 .. n-R+r, or the last W of them with a sliding window):
//     s_j = (q . k^_j) * sm_scale,   k^_j = decode(codeK_j) * scaleK_j,   v^_j likewise,   o = softmax(s) v^.
//
// One CTA = (KV head, request, key slice), in that grid order (the KV heads of a slice side by side; every
// request's first slices before the short last ones, so the last wave holds short work): its R x G query
// rows (R <= 8 rows, G <= 8 query heads of the KV head) are the M = 128 rows of the products, the keys of the
// slice come in tiles of 128.
//  * QK^T on the stored codes: the K codes are copied as they are (cp.async) into the 128-byte-swizzled
//    K-major tile that kind::f8f6f4 MMAs read.  The query row is brought to |x| < 256 by a power of two
//    (x = q 2^(7-e), e the exponent of the row's largest element) and split into two E4M3 pieces,
//    x = hi + lo with lo = E4M3(x - hi): error at most 2^-8 |x| + 2^-10 against max |x| >= 128.  S = hi K^T +
//    lo K^T accumulates exact E4M3 products in FP32 in TMEM; the softmax takes
//    s = S * scaleK * 2^(e-7) * sm_scale * log2(e).
//  * PV on FP16: E4M3 codes convert exactly to FP16, so the V tile holds the stored codes as FP16 (the V codes
//    land in a staging ring and are converted in shared memory) and the V scale stays out of the product.
//  * The V scale goes into the probabilities: w = 2^(s - m) * scaleV.  FP16 has a narrow exponent range and the
//    per-row V scales of a slice can span 2^30, so P' = w 2^-E with one power-of-two exponent E per row that only
//    grows (raised when some w would exceed 2^(E + 12)); the maximum m is lazy (raised when a score exceeds it by
//    more than 8).  Either raise rescales the row of O in TMEM (rare); O is in units of 2^E.  The sign of
//    sm_scale goes into the query pieces, so the multiplier of S is positive.
//  * Rows and lane quarters.  A warp reaches only its own quarter of the TMEM lanes (32 (w % 4) .. +31), so a
//    request of up to 32 live rows would leave three SM sub-partitions idle.  The Q tile therefore repeats the
//    live rows in every quarter (one row group of 32 rows in all four, or two groups of 32 in two quarters
//    each), and each quarter takes its own share of every tile's key columns (32 or 64): it keeps its own
//    maximum, sum, exponent and rows of O (its PV product sees P' = 0 outside its columns), and the quarters of
//    a row are merged like split-K partials at the end of the slice.
//  * Warps: 0-3 softmax (one per lane quarter, one query row per thread), 4 the MMA issuer (lane 0) and owner of
//    the TMEM allocation, 5-8 the K copy warps, 9-12 the V copy warps (13 warps: at most 128 registers a
//    thread).  A copy lane copies one 16-byte part of the rows of 8 keys per tile (lanes 8k .. 8k+7 share a
//    key's 128-byte row) with cp.async, which lands in shared memory without passing through L1: loads into
//    registers stalled behind the small L1 left next to ~215 KB of shared memory (64-request batch: 1,590 us
//    with register loads and FP16 K, 996 us with cp.async and E4M3 K).  The gather rate follows the number of
//    warps issuing copies: two copy warps per tensor 897 us, four 757 us, eight (80 registers a thread, the
//    softmax spilling) 1,007 us.
//    Rings: K 4 x 16 KB (E4M3, read by the MMA as it lands), V codes 3 x 16 KB, V FP16 2 x 32 KB (MN-major,
//    written by the V copy lanes from their own staged chunks), scales 6 x 1 KB.  Lanes of the K warps also
//    copy both scales of the tile's keys into their ring, which the softmax releases, so the softmax never
//    waits for a V tile.
//  * TMEM: S0, S1 (128 columns each, double buffered), O (128), P0, P1 (64 columns of FP16 pairs).
//  * The split merge: the CTA whose slice of (request, KV head) finishes last merges all slices (decode_merge.cuh).
// Every mbarrier wait is bounded in time; on expiry the CTA flags an error, drains and exits.
#include <cfloat>
#include <mutex>
#include <type_traits>

#include "decode_common.cuh"
#include "decode_merge.cuh"
#include "ftkv_device.cuh"
#include "ftkv_internal.h"

namespace ftkv {
namespace {

constexpr int MR_BN = 128;   // keys per tile
constexpr uint32_t MR_BOX = 128 * 128;         // one 128-row x 128-byte swizzle box: 128 E4M3 or 64 FP16 a row
constexpr uint32_t MR_TILE = 2 * MR_BOX;       // FP16 V tile: 128 keys x 128 FP16
// ring stages: K (E4M3 codes, read by the MMA as they land), V codes as they land, V as FP16, scales
constexpr int MR_NSK = 4, MR_NSR = 3, MR_NSV = 2, MR_NSC = 6;
constexpr int MR_DK = 2, MR_DV = 2;  // tiles whose copies stay in flight while a copy warp completes the oldest
constexpr uint32_t MR_OFF_Q = 0;                             // Q high and low E4M3 pieces (one box each)
constexpr uint32_t MR_OFF_K = MR_OFF_Q + 2 * MR_BOX;
constexpr uint32_t MR_OFF_R = MR_OFF_K + MR_NSK * MR_BOX;
constexpr uint32_t MR_OFF_V = MR_OFF_R + MR_NSR * MR_BOX;
constexpr uint32_t MR_SC_FLOATS = 2 * 128;                 // per scale stage: K scales, V scales
constexpr uint32_t MR_OFF_SC = MR_OFF_V + MR_NSV * MR_TILE;
constexpr uint32_t MR_OFF_X = MR_OFF_SC + MR_NSC * MR_SC_FLOATS * 4;   // quarters' (m, l) exchange [4][32][2]
constexpr uint32_t MR_OFF_BAR = MR_OFF_X + 4 * 32 * 2 * 4;
constexpr int MR_B_QFULL = 0, MR_B_KFULL0 = 1, MR_B_KEMPTY0 = 5, MR_B_VFULL0 = 9, MR_B_VEMPTY0 = 11,
              MR_B_SFULL0 = 13, MR_B_SFREE0 = 15, MR_B_PFULL0 = 17, MR_B_ODONE = 19, MR_B_OFINAL = 20,
              MR_B_DRAIN = 21, MR_B_CFULL0 = 22, MR_B_CEMPTY0 = 28, MR_NBAR = 34;
constexpr uint32_t MR_SCRATCH = MR_NSK * MR_BOX + MR_NSR * MR_BOX + MR_NSV * MR_TILE;  // rings, free at the end
constexpr uint32_t MR_OFF_MISC = MR_OFF_BAR + MR_NBAR * 8;  // TMEM base address, abort flag
constexpr uint32_t MR_SMEM = MR_OFF_MISC + 16 + 1024;       // + slack for the 1024-byte alignment
static_assert(MR_SMEM <= 232448, "decode_mr shared memory");
constexpr uint32_t MR_TMEM_COLS = 512;
constexpr uint32_t MR_TMEM_O = 256, MR_TMEM_P = 384;
constexpr int MR_CW = 4;                            // copy warps per tensor (K, V)
constexpr int MR_THREADS = (5 + 2 * MR_CW) * 32;
constexpr int MR_MMA_WARP = 4, MR_KW0 = 5, MR_VW0 = 5 + MR_CW;  // the MMA warp, the first K and the first V copy warp
constexpr int MR_CL = 32 * MR_CW;                   // copy lanes per tensor
constexpr int MR_KPR = MR_CL / 8;                   // keys per copy round (8 lanes per 128-byte row)
constexpr int MR_RND = MR_BN / MR_KPR;              // rounds per tile
constexpr int MR_SPL = (MR_RND + 7) / 8;            // slots held per lane (lanes past MR_RND / MR_SPL hold none)
static_assert(MR_RND * MR_KPR == MR_BN && (MR_RND <= 8 || MR_RND % 8 == 0), "copy lanes");
constexpr unsigned long long MR_WAIT_NS = 2000000000ull;
constexpr float kMrLazyMax = 8.0f;
constexpr int kMrLazyExp = 12;

// Byte offset of 16-byte chunk c (8 FP16 of d = 8c .. 8c+7) of row r in a 128-byte-swizzled tile of 128 rows x
// 128 FP16 (two 64-column boxes).
__device__ __forceinline__ uint32_t mr_chunk(int r, int c) {
  return (c >> 3) * MR_BOX + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}
// Byte offset of 16-byte chunk c (16 E4M3 of d = 16c .. 16c+15) of row r in a 128-byte-swizzled box of 128 rows.
__device__ __forceinline__ uint32_t mr_chunk8(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// tcgen05 shared-memory matrix descriptor: start, leading / stride byte offsets, 128-byte swizzle.
__device__ __forceinline__ uint64_t mr_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;  // swizzle: 128 bytes
  return d;
}
// K-major E4M3 box, k-step kk (32 columns); MN-major FP16 V tile (keys x d, d contiguous), k-step kk = keys 16kk ..
__device__ __forceinline__ uint64_t mr_kdesc(uint32_t box, int kk) { return mr_desc(box + kk * 32, 16, 1024); }
__device__ __forceinline__ uint64_t mr_vdesc(uint32_t tile, int kk) { return mr_desc(tile + kk * 2048, MR_BOX, 1024); }

// Instruction descriptor, M = 128, N = 128, FP32 accumulate; A and B types 0 (FP16 for kind::f16, E4M3 for
// kind::f8f6f4).
__host__ __device__ constexpr uint32_t mr_idesc(bool b_mn_major) {
  return (1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
}

// D += A B, A and B E4M3 in shared memory
__device__ __forceinline__ void mr_mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D += A B with A read from tensor memory (128 lanes = rows, 8 columns = 16 FP16 of K)
__device__ __forceinline__ void mr_mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mr_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mr_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void mr_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// generic-proxy writes to shared memory become visible to the tensor cores (async proxy)
__device__ __forceinline__ void mr_fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void mr_tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void mr_tmem_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]),
      "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]),
      "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]),
      "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}
__device__ __forceinline__ void mr_tmem_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void mr_tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void mr_tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mr_bar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mr_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mr_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity; false (abort flag and device error raised) on expiry or when
// another thread aborted.
__device__ __noinline__ bool mr_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err) {
  if (mr_try_wait(bar, parity)) return true;
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  while (true) {
    if (mr_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    __nanosleep(128);  // a waiting warp gives its issue slots to the warps that compute
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > MR_WAIT_NS) {
      *abort_flag = 1;
      flag_error(err, kDevErrTimeout);
      return false;
    }
  }
}

// 8 E4M3 codes (two words) -> 8 FP16 (one 16-byte chunk), exact
__device__ __forceinline__ uint4 mr_codes_to_f16(uint32_t w0, uint32_t w1) {
  return make_uint4(e4m3_lo2(w0), e4m3_hi2(w0), e4m3_lo2(w1), e4m3_hi2(w1));
}

__global__ void __launch_bounds__(MR_THREADS, 1) decode_mr_kernel(const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + MR_OFF_MISC + 4);
  auto bar = [&](int i) { return base + MR_OFF_BAR + 8u * i; };

  griddep_launch_dependents();
  griddep_wait();
  const int h = blockIdx.x, b = blockIdx.y, split = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.group;

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
  if (R == 0) return;
  if (n == 0) {  // no keys: the rows of this KV head's group are zero
    if (split == 0)
      for (int i = threadIdx.x; i < R * G * kHeadDim; i += blockDim.x)
        a.out[((row0 + i / (G * kHeadDim)) * a.num_q_heads + h * G + (i / kHeadDim) % G) * kHeadDim + i % kHeadDim] = 0;
    return;
  }
  const int kfirst = static_cast<int>(first_key(a, n, R));  // slices cover keys [kfirst, n)
  const int j0 = kfirst + split * static_cast<int>(a.chunk);
  const int j1 = (static_cast<int64_t>(j0) + a.chunk < n) ? j0 + static_cast<int>(a.chunk) : static_cast<int>(n);
  if (j0 >= n) return;  // slices past the end hold no keys and take no ticket
  const int T = (j1 - j0 + MR_BN - 1) / MR_BN;  // key tiles of the slice
  const int nrows = R * G;  // live query rows (<= 64)

  // ---- fused store: the request's new tokens (positions n-R .. n-1) that fall in this slice are quantized into
  // the pool first (one warp per token: K row on lanes 0-15, V row on 16-31, the store kernel's arithmetic); the
  // barrier below orders these writes before every copy warp's loads, which then read the new rows like any other
  // key ----
  if (a.k_new) {
    const int nq0 = static_cast<int>(n) - R;  // position of the request's first new token
    const int first = (nq0 > j0) ? nq0 : j0;
    bool wrote = false;
    for (int pos = first + warp; pos < j1; pos += MR_THREADS / 32) {  // warp-uniform
      const int half = lane >> 4, l = lane & 15;
      const uint16_t* src = (half ? a.v_new : a.k_new) + ((row0 + pos - nq0) * a.num_kv_heads + h) * kHeadDim + l * 8;
      const uint4 rawv = __ldg(reinterpret_cast<const uint4*>(src));
      const int32_t sv = a.req_to_slot[static_cast<int64_t>(b) * a.req_stride + pos];
      float sc;
      const uint2 packed = quantize_row_lane8(rawv, sc);
      if (sv >= 0 && sv < a.num_rows) {  // a bad slot is flagged by the copy warps; nothing is written
        const int64_t row = static_cast<int64_t>(sv) * a.num_kv_heads + h;
        *reinterpret_cast<uint2*>(const_cast<uint8_t*>(half ? a.v_codes : a.k_codes) + row * kHeadDim + l * 8) = packed;
        if (l == 0) const_cast<float*>(half ? a.v_scales : a.k_scales)[row] = sc;
      }
      wrote = true;
    }
    if (wrote) __threadfence();  // the rows reach L2 before the barrier below
  }

  if (threadIdx.x == 0) {
    mr_bar_init(bar(MR_B_QFULL), 128);
    for (int s = 0; s < MR_NSK; s++) {
      mr_bar_init(bar(MR_B_KFULL0 + s), MR_CL);
      mr_bar_init(bar(MR_B_KEMPTY0 + s), 1);
    }
    for (int s = 0; s < MR_NSV; s++) {
      mr_bar_init(bar(MR_B_VFULL0 + s), MR_CL);
      mr_bar_init(bar(MR_B_VEMPTY0 + s), 1);
    }
    for (int s = 0; s < 2; s++) {
      mr_bar_init(bar(MR_B_SFULL0 + s), 1);
      mr_bar_init(bar(MR_B_SFREE0 + s), 4);  // one lane of each softmax warp
      mr_bar_init(bar(MR_B_PFULL0 + s), 4);
    }
    for (int s = 0; s < MR_NSC; s++) {
      mr_bar_init(bar(MR_B_CFULL0 + s), 2 * MR_KPR);  // the scale lanes (when their copies land)
      mr_bar_init(bar(MR_B_CEMPTY0 + s), 4);
    }
    mr_bar_init(bar(MR_B_ODONE), 1);
    mr_bar_init(bar(MR_B_OFINAL), 1);
    mr_bar_init(bar(MR_B_DRAIN), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the scale ring starts at zero: the softmax multiplies every column, including keys past the slice whose
  // scales are never copied, by a finite scale
  for (int i = threadIdx.x; i < MR_NSC * MR_SC_FLOATS; i += MR_THREADS)
    reinterpret_cast<float*>(gbase + MR_OFF_SC)[i] = 0.0f;
  if (warp == MR_MMA_WARP) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(base + MR_OFF_MISC),
                 "r"(MR_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  mr_fence_before();
  __syncthreads();
  mr_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + MR_OFF_MISC);

  float lsum = 0.0f, mrow = -INFINITY;  // softmax threads: running sum and (lazy) maximum of their row
  int Erow = -126;                      // FP16 operand exponent of the row: P' = w 2^-E

  // ---------------- query tile, then softmax: warp lg owns TMEM lanes 32 lg .. +31 ----------------
  // NSW row groups of 32 query rows (1 for up to 32 live rows, else 2).  Lane quarter lg holds rows 32 rg .. +31
  // (rg = lg % NSW) and takes key columns CW kp .. +CW-1 of every tile (kp = lg / NSW, CW = 32 NSW): the Q tile
  // repeats the live rows in every quarter, so the softmax runs on all four SM sub-partitions, and each quarter
  // keeps its own maximum, sum, exponent and O (its PV product sees P' = 0 outside its key columns).  The
  // quarters of a row are merged at the end of the slice.
  auto softmax = [&](auto nsw_c) {
    constexpr int NSW = decltype(nsw_c)::value;
    constexpr int NQ = 4 / NSW;   // key slices of a tile
    constexpr int CW = 128 / NQ;  // key columns of a tile per softmax warp
    const int lg = warp, rg = lg % NSW, kp = lg / NSW;
    const int qrow = rg * 32 + lane;  // query row r G + head of the request
    const bool live = qrow < nrows;
    const int rr = live ? qrow / G : 0, hq = live ? qrow % G : 0;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(lg * 32) << 16);
    auto softmax_sync = [&]() { asm volatile("bar.sync 1, 128;" ::: "memory"); };
    // Q row -> x = q 2^(7-e) (|x| < 256), split into E4M3 pieces x = hi + lo (lo = E4M3(x - hi): the error is at
    // most 2^-8 |x| + 2^-10, against max |x| >= 128), written as M row 32 lg + lane of the two K-major swizzled
    // boxes (zeros past nrows)
    float qmul = 0.0f;
    {
      uint4 qv[16];
      const uint4* src = reinterpret_cast<const uint4*>(a.q + ((row0 + rr) * a.num_q_heads + h * G + hq) * kHeadDim);
#pragma unroll
      for (int c = 0; c < 16; c++) qv[c] = live ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
      float amax = 0.0f;
#pragma unroll
      for (int c = 0; c < 16; c++) {
        const uint32_t w[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
#pragma unroll
        for (int e = 0; e < 4; e++) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[e])), fabsf(bf16_hi(w[e]))));
      }
      int ex = (amax > 0.0f) ? ilogbf(amax) : 0;
      ex = ex < -120 ? -120 : ex;
      // the sign of the softmax scale goes into the pieces (exact), so the multiplier qmul is positive
      const float up = copysignf(__uint_as_float(static_cast<uint32_t>(127 + 7 - ex) << 23), a.qk_scale_log2);
      // (> 0: a zero softmax scale still gives finite products s' qmul and -inf for the masked columns)
      qmul = fmaxf(__uint_as_float(static_cast<uint32_t>(127 - 7 + ex) << 23) * fabsf(a.qk_scale_log2), FLT_MIN);
      const int m = lg * 32 + lane;
#pragma unroll
      for (int c = 0; c < 8; c++) {  // 16 d per chunk: two uint4 of BF16
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const uint32_t w0 = (e < 2) ? (e == 0 ? qv[2 * c].x : qv[2 * c].z) : (e == 2 ? qv[2 * c + 1].x : qv[2 * c + 1].z);
          const uint32_t w1 = (e < 2) ? (e == 0 ? qv[2 * c].y : qv[2 * c].w) : (e == 2 ? qv[2 * c + 1].y : qv[2 * c + 1].w);
          const float x0 = bf16_lo(w0) * up, x1 = bf16_hi(w0) * up, x2 = bf16_lo(w1) * up, x3 = bf16_hi(w1) * up;
          const uint32_t h01 = e4m3x2_encode(x0, x1), h23 = e4m3x2_encode(x2, x3);
          const float2 b01 = f16x2_to_float2(e4m3x2_to_f16x2(h01)), b23 = f16x2_to_float2(e4m3x2_to_f16x2(h23));
          const uint32_t l01 = e4m3x2_encode(x0 - b01.x, x1 - b01.y), l23 = e4m3x2_encode(x2 - b23.x, x3 - b23.y);
          hw[e] = h01 | (h23 << 16);
          lw[e] = l01 | (l23 << 16);
        }
        st_shared_v4(base + MR_OFF_Q + mr_chunk8(m, c), make_uint4(hw[0], hw[1], hw[2], hw[3]));
        st_shared_v4(base + MR_OFF_Q + MR_BOX + mr_chunk8(m, c), make_uint4(lw[0], lw[1], lw[2], lw[3]));
      }
      mr_fence_async_smem();
      mr_arrive(bar(MR_B_QFULL));
    }
    // both P buffers of this quarter: zero once; every tile then writes only the quarter's own key columns
    {
      const uint32_t z[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
      for (int c = 0; c < 128; c += 16) mr_tmem_st16(lane_base + MR_TMEM_P + c, z);
      mr_tmem_st_wait();
    }
    // visible keys of this row: [low, vis) (and the slice [j0, j1))
    const int vis = static_cast<int>(n) - R + rr + 1;
    const int low = (a.window > 0 && vis - a.window > 0) ? vis - static_cast<int>(a.window) : 0;
    const int lo = low > j0 ? low : j0, hi = vis < j1 ? vis : j1;
    float wlim = exp2i(-126 + kMrLazyExp), iw = exp2i(126);
    const int cb = kp * CW;  // this warp's first key column
    bool ok = true;
    for (int j = 0; j < T; j++) {
      const int bb = j & 1, sc = j % MR_NSC;
      if (ok) ok = __all_sync(0xffffffffu, mr_wait(bar(MR_B_SFULL0 + bb), (j >> 1) & 1, abort_flag, a.err));
      if (ok) ok = __all_sync(0xffffffffu, mr_wait(bar(MR_B_CFULL0 + sc), (j / MR_NSC) & 1, abort_flag, a.err));
      if (!ok) break;
      const float* ks = reinterpret_cast<const float*>(gbase + MR_OFF_SC + sc * MR_SC_FLOATS * 4) + cb;
      const float* vs = ks + MR_BN;
      const int kb = j0 + j * MR_BN + cb;
      const int c0 = lo - kb, c1 = hi - kb;  // visible columns [c0, c1) of this warp's CW
      const bool full = __all_sync(0xffffffffu, c0 <= 0 && c1 >= CW);
      const uint32_t sb = lane_base + bb * 128 + cb;
      // pass 1: s' = S scaleK and its maximum (four partial maxima: the warp is alone on its sub-partition, so the
      // chains' latency is not hidden by other warps); s = s' qmul, qmul > 0
      float sv[CW];  // this warp's columns of S, all loads in flight at once
      mr_fence_after();
#pragma unroll
      for (int q = 0; q < CW / 32; q++) mr_tmem_ld32(sb + 32 * q, sv + 32 * q);
      mr_tmem_ld_wait();
      mr_fence_before();
      __syncwarp();
      if (lane == 0) mr_arrive(bar(MR_B_SFREE0 + bb));  // S buffer bb read: free for the QK product of tile j + 2
#pragma unroll
      for (int e4 = 0; e4 < CW / 4; e4++) {
        const float4 k4 = *reinterpret_cast<const float4*>(ks + 4 * e4);
        sv[4 * e4] *= k4.x;
        sv[4 * e4 + 1] *= k4.y;
        sv[4 * e4 + 2] *= k4.z;
        sv[4 * e4 + 3] *= k4.w;
      }
      if (!full) {  // the slice's boundary tiles: columns outside the row's visible keys drop out
#pragma unroll
        for (int c = 0; c < CW; c++) sv[c] = (c >= c0 && c < c1) ? sv[c] : -INFINITY;
      }
      float tm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < CW; c++) tm[c & 3] = fmaxf(tm[c & 3], sv[c]);
      const float tmax = fmaxf(fmaxf(tm[0], tm[1]), fmaxf(tm[2], tm[3])) * qmul;
      // lazy maximum and FP16 exponent; f rescales O (and l: fm)
      float fm = 1.0f;
      if (tmax > mrow + kMrLazyMax) {
        fm = (mrow == -INFINITY) ? 1.0f : fast_exp2(mrow - tmax);
        mrow = tmax;
        lsum *= fm;
      }
      const float sub = (mrow == -INFINITY) ? 0.0f : mrow;
      // pass 2: p = 2^(s - m) (summed), w = p scaleV (kept in sv) and the tile's largest w
      // (a key past the slice has p = 0 and a finite stale or zero scale in the ring)
      float pa[4] = {0.0f, 0.0f, 0.0f, 0.0f}, wa[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int e4 = 0; e4 < CW / 4; e4++) {
        const float4 v4 = *reinterpret_cast<const float4*>(vs + 4 * e4);
        const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const int c = 4 * e4 + e;
          const float p = fast_exp2(fmaf(sv[c], qmul, -sub));
          pa[e] += p;
          sv[c] = p * vv[e];
          wa[e] = fmaxf(wa[e], sv[c]);
        }
      }
      lsum += (pa[0] + pa[1]) + (pa[2] + pa[3]);
      const float wbound = fmaxf(fmaxf(wa[0], wa[1]), fmaxf(wa[2], wa[3]));
      float fe = 1.0f;
      if (wbound > wlim) {  // raise E (an exact power of two; E never decreases)
        const int e0 = max(Erow, max(static_cast<int>(__float_as_uint(wbound) >> 23), 1) - 127);
        const int ne = min(e0, 127 - kMrLazyExp);
        fe = (Erow - ne < -126) ? 0.0f : exp2i(Erow - ne);
        Erow = ne;
        wlim = exp2i(ne + kMrLazyExp);
        iw = exp2i(-ne);
      }
      const float f = fm * fe;
      if (__any_sync(0xffffffffu, f != 1.0f) && j >= 1) {
        // O holds PV_0 .. PV_{j-1}: wait for the last of them, then scale this quarter's rows of O in place
        ok = __all_sync(0xffffffffu, mr_wait(bar(MR_B_ODONE), (j - 1) & 1, abort_flag, a.err));
        if (!ok) break;
        mr_fence_after();
#pragma unroll 1
        for (int q = 0; q < 4; q++) {
          float o[32];
          mr_tmem_ld32(lane_base + MR_TMEM_O + q * 32, o);
          mr_tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; e++) o[e] *= f;
          mr_tmem_st32(lane_base + MR_TMEM_O + q * 32, o);
        }
        mr_tmem_st_wait();
      }
      // pass 3: P' = w 2^-E as FP16 pairs into this warp's columns of P buffer bb
#pragma unroll
      for (int q = 0; q < CW / 32; q++) {
        uint32_t pw[16];
#pragma unroll
        for (int e2 = 0; e2 < 16; e2++) {
          const __half2 hv = __floats2half2_rn(sv[q * 32 + 2 * e2] * iw, sv[q * 32 + 2 * e2 + 1] * iw);
          pw[e2] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        mr_tmem_st16(lane_base + MR_TMEM_P + bb * 64 + cb / 2 + q * 16, pw);
      }
      mr_tmem_st_wait();
      mr_fence_before();
      __syncwarp();
      if (lane == 0) {
        mr_arrive(bar(MR_B_CEMPTY0 + sc));  // the tile's scales are read
        mr_arrive(bar(MR_B_PFULL0 + bb));
      }
    }
    // ---- epilogue: the NQ quarters of each row merged into this slice's partial (m, l, O in units of 2^m) ----
    const bool fin = ok && __all_sync(0xffffffffu, mr_wait(bar(MR_B_OFINAL), 0, abort_flag, a.err));
    float2* xq = reinterpret_cast<float2*>(gbase + MR_OFF_X);  // [4 quarters][32 lanes]: (m, l)
    xq[lg * 32 + lane] = make_float2(mrow, lsum);
    softmax_sync();
    float M = -INFINITY, L = 0.0f;
#pragma unroll
    for (int k = 0; k < NQ; k++) M = fmaxf(M, xq[(rg + k * NSW) * 32 + lane].x);
#pragma unroll
    for (int k = 0; k < NQ; k++) {
      const float2 t = xq[(rg + k * NSW) * 32 + lane];
      L += (t.x == -INFINITY) ? 0.0f : t.y * fast_exp2(t.x - M);
    }
    // O rows of the quarters, scaled to units of 2^M, staged in the free rings: [NQ][32 NSW rows][132 floats]
    float* red = reinterpret_cast<float*>(gbase + MR_OFF_K);
    if (fin) {
      const float g = (mrow == -INFINITY) ? 0.0f : fast_exp2(mrow - M) * exp2i(Erow);
      float4* dst = reinterpret_cast<float4*>(red + (kp * 32 * NSW + qrow) * 132);
      mr_fence_after();
#pragma unroll 1
      for (int q = 0; q < 4; q++) {
        float o[32];
        mr_tmem_ld32(lane_base + MR_TMEM_O + q * 32, o);
        mr_tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 8; e++) dst[q * 8 + e] = make_float4(o[4 * e] * g, o[4 * e + 1] * g, o[4 * e + 2] * g, o[4 * e + 3] * g);
      }
    }
    softmax_sync();
    if (fin) {
      // warp w writes d = 32 w + lane of every live row (128-byte rows of the partial)
      const int d = 32 * warp + lane;
      for (int r = 0; r < nrows; r++) {
        float acc = 0.0f;
#pragma unroll
        for (int k = 0; k < NQ; k++) acc += red[(k * 32 * NSW + r) * 132 + d];
        const int64_t prow = ((row0 + r / G) * a.num_q_heads + h * G + r % G) * a.num_splits * a.pps + split;
        a.part_acc[prow * kHeadDim + d] = acc;
      }
      if (kp == 0 && live) {
        const int64_t prow = ((row0 + rr) * a.num_q_heads + h * G + hq) * a.num_splits * a.pps + split;
        a.part_ml[prow * 2] = M;
        a.part_ml[prow * 2 + 1] = L;
      }
    }
  };

  if (warp < 4) {
    if (nrows <= 32)
      softmax(std::integral_constant<int, 1>{});
    else
      softmax(std::integral_constant<int, 2>{});
  } else if (warp == MR_MMA_WARP) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t IDESC_QK = mr_idesc(false);  // kind::f8f6f4, E4M3 x E4M3
      constexpr uint32_t IDESC_PV = mr_idesc(true);
      bool ok = mr_wait(bar(MR_B_QFULL), 0, abort_flag, a.err);
      auto issue_pv = [&](int i) -> bool {
        const int bb = i & 1, sv = i % MR_NSV;
        if (!mr_wait(bar(MR_B_PFULL0 + bb), (i >> 1) & 1, abort_flag, a.err)) return false;
        if (!mr_wait(bar(MR_B_VFULL0 + sv), (i / MR_NSV) & 1, abort_flag, a.err)) return false;
        mr_fence_after();
        const uint32_t vt = base + MR_OFF_V + sv * MR_TILE;
#pragma unroll
        for (int kk = 0; kk < 8; kk++)
          mr_mma_ta(tmem + MR_TMEM_O, tmem + MR_TMEM_P + bb * 64 + kk * 8, mr_vdesc(vt, kk), IDESC_PV,
                    (i > 0 || kk > 0) ? 1u : 0u);
        mr_commit(bar(MR_B_VEMPTY0 + sv));
        mr_commit(bar(MR_B_ODONE));
        return true;
      };
      for (int j = 0; ok && j < T; j++) {
        const int bb = j & 1, sk = j % MR_NSK;
        if (!mr_wait(bar(MR_B_KFULL0 + sk), (j / MR_NSK) & 1, abort_flag, a.err)) { ok = false; break; }
        if (j >= 2 && !mr_wait(bar(MR_B_SFREE0 + bb), ((j >> 1) - 1) & 1, abort_flag, a.err)) { ok = false; break; }
        mr_fence_after();
        const uint32_t kt = base + MR_OFF_K + sk * MR_BOX;
#pragma unroll
        for (int pc = 0; pc < 2; pc++)  // S = Q_hi K^T + Q_lo K^T
#pragma unroll
          for (int kk = 0; kk < 4; kk++)
            mr_mma_f8(tmem + bb * 128, mr_kdesc(base + MR_OFF_Q + pc * MR_BOX, kk), mr_kdesc(kt, kk), IDESC_QK,
                      (pc > 0 || kk > 0) ? 1u : 0u);
        mr_commit(bar(MR_B_SFULL0 + bb));
        mr_commit(bar(MR_B_KEMPTY0 + sk));  // K tile j is consumed once its QK product is done
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok && issue_pv(T - 1)) mr_commit(bar(MR_B_OFINAL));
      // drain every MMA issued by this thread before TMEM is released
      mr_commit(bar(MR_B_DRAIN));
      mr_wait(bar(MR_B_DRAIN), 0, abort_flag, a.err);
    }
  } else {
    // ---------------- copy warps: MR_CW for K, then MR_CW for V; MR_RND cp.async of 16 bytes a lane and tile -------
    // Lane (kr, part) copies 16-byte part `part` of the rows of keys KPR r + kr, r < MR_RND.  K codes land directly in
    // the 128-byte-swizzled box the MMA reads; V codes land in a plain ring and the same lane converts its own
    // chunks to FP16.  A warp keeps MR_DK (MR_DV) tiles in flight while it completes the oldest: it waits for its
    // own copies of that tile, makes them visible to the tensor cores and arrives on the tile's barrier.
    const bool is_v = warp >= MR_VW0;
    const int cl = (warp - (is_v ? MR_VW0 : MR_KW0)) * 32 + lane;
    const int kr = cl >> 3, part = cl & 7;  // key within a round of MR_KPR, 16-byte part of the row
    const uint8_t* codes = is_v ? a.v_codes : a.k_codes;
    const int64_t hkv = a.num_kv_heads;
    const bool scl_lane = !is_v && part < 2;  // K lanes of part 0 / 1: the K / V scales of their keys
    const float* scales = part ? a.v_scales : a.k_scales;
    const int32_t* srow = a.req_to_slot + static_cast<int64_t>(b) * a.req_stride;
    // codes are read once: their L2 lines go first, and the 32-byte scale sectors, which the CTAs of the other
    // KV heads of the slice read too, stay longer (64-request batch: 710 us against 715)
    const uint64_t pol_codes = l2_policy_evict_first();
    // slots of keys kb + KPR r + kr of tile jt, r = SPL part + i: the 8 lanes of a key group hold the MR_RND slots
    // of its keys between them (loaded a tile ahead of their use; checked where used)
    auto load_slots = [&](int jt, int32_t (&sl)[MR_SPL]) {
      const int kb = j0 + jt * MR_BN;
#pragma unroll
      for (int i = 0; i < MR_SPL; i++) {
        const int rd = MR_SPL * part + i;
        const int key = kb + MR_KPR * rd + kr;
        sl[i] = (rd < MR_RND && key < j1) ? __ldg(srow + key) : 0;
      }
    };
    // cp.async of tile jt's codes (and, on the scale lanes, its scales: stage jt % MR_NSC of the scale ring,
    // released by the softmax of tile jt - MR_NSC; its barrier is arrived on when they land); one group per tile
    auto issue = [&](int jt, int32_t (&sl)[MR_SPL]) -> bool {
      const int kb = j0 + jt * MR_BN;
      bool bad = false;
#pragma unroll
      for (int i = 0; i < MR_SPL; i++) {
        bad |= sl[i] < 0 || sl[i] >= a.num_rows;
        sl[i] = (sl[i] < 0 || sl[i] >= a.num_rows) ? 0 : sl[i];
      }
      if (bad) flag_error(a.err, kDevErrBadSlot);
      bool okw = true;
      if (!is_v && jt >= MR_NSK)  // K box jt % MR_NSK: free once the QK product of tile jt - MR_NSK is done
        okw = mr_wait(bar(MR_B_KEMPTY0 + jt % MR_NSK), (jt / MR_NSK - 1) & 1, abort_flag, a.err);
      const int c = jt % MR_NSC, uc = jt / MR_NSC;
      if (okw && scl_lane && uc >= 1) okw = mr_wait(bar(MR_B_CEMPTY0 + c), (uc - 1) & 1, abort_flag, a.err);
      if (!__all_sync(0xffffffffu, okw)) return false;
      const uint32_t box = is_v ? base + MR_OFF_R + (jt % MR_NSR) * MR_BOX : base + MR_OFF_K + (jt % MR_NSK) * MR_BOX;
      const uint32_t dsc = base + MR_OFF_SC + (c * MR_SC_FLOATS + part * MR_BN) * 4;
#pragma unroll
      for (int r = 0; r < MR_RND; r++) {
        const int32_t slot = __shfl_sync(0xffffffffu, sl[r % MR_SPL], (lane & ~7) | (r / MR_SPL));
        const int key = MR_KPR * r + kr;
        const int64_t row = static_cast<int64_t>(slot) * hkv + h;
        const uint32_t dst = box + (is_v ? key * 128 + part * 16 : mr_chunk8(key, part));
        if (kb + key < j1) {
          cp_async_16_hint(dst, codes + row * kHeadDim + part * 16, pol_codes);
          if (scl_lane) cp_async_4(dsc + key * 4, scales + row);
        } else if (!is_v) {
          st_shared_v4(dst, make_uint4(0u, 0u, 0u, 0u));  // keys past the slice: zero rows of K
        }
      }
      if (scl_lane)
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar(MR_B_CFULL0 + c)) : "memory");
      asm volatile("cp.async.commit_group;" ::: "memory");
      return true;
    };
    // wait for this lane's copies of tile t, with `newer` younger groups left in flight
    auto wait_tile = [&](int newer) {
      static_assert(MR_DK <= 3 && MR_DV <= 3, "cp.async groups in flight");
      if (newer >= 3)
        asm volatile("cp.async.wait_group 3;" ::: "memory");
      else if (newer == 2)
        asm volatile("cp.async.wait_group 2;" ::: "memory");
      else if (newer == 1)
        asm volatile("cp.async.wait_group 1;" ::: "memory");
      else
        asm volatile("cp.async.wait_group 0;" ::: "memory");
    };
    // tile t has landed: K -> visible to the MMA; V -> converted to FP16 into stage t % MR_NSV (free once the PV
    // product of tile t - MR_NSV is done)
    auto complete = [&](int t) -> bool {
      if (!is_v) {
        mr_fence_async_smem();
        mr_arrive(bar(MR_B_KFULL0 + t % MR_NSK));
        return true;
      }
      const int sv = t % MR_NSV;
      bool okw = true;
      if (t >= MR_NSV) okw = mr_wait(bar(MR_B_VEMPTY0 + sv), (t / MR_NSV - 1) & 1, abort_flag, a.err);
      if (!__all_sync(0xffffffffu, okw)) return false;
      const int kb = j0 + t * MR_BN;
      const uint32_t raw = base + MR_OFF_R + (t % MR_NSR) * MR_BOX;
      const uint32_t st = base + MR_OFF_V + sv * MR_TILE;
#pragma unroll
      for (int r = 0; r < MR_RND; r++) {
        const int key = MR_KPR * r + kr;
        const uint4 d = (kb + key < j1) ? ld_shared_v4(raw + key * 128 + part * 16) : make_uint4(0u, 0u, 0u, 0u);
        st_shared_v4(st + mr_chunk(key, 2 * part), mr_codes_to_f16(d.x, d.y));
        st_shared_v4(st + mr_chunk(key, 2 * part + 1), mr_codes_to_f16(d.z, d.w));
      }
      mr_fence_async_smem();
      mr_arrive(bar(MR_B_VFULL0 + sv));
      return true;
    };
    const int D = is_v ? MR_DV : MR_DK;
    int32_t slots[MR_SPL];
    load_slots(0, slots);
    for (int jt = 0; jt < T + D; jt++) {
      if (jt < T) {
        if (!issue(jt, slots)) break;
        load_slots(jt + 1, slots);
      }
      const int t = jt - D;
      if (t >= 0) {
        wait_tile((jt < T ? jt : T - 1) - t);
        if (!complete(t)) break;
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // no copy outlives the CTA's shared memory
  }

  mr_fence_before();
  __syncthreads();
  if (warp == MR_MMA_WARP) {
    mr_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(MR_TMEM_COLS) : "memory");
  }
  if (*abort_flag) return;

  // ---- split merge, done by the last slice of (request, KV head) to arrive ----
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
  merge_split_partials(a, row0, R, h, nslices, gbase + MR_OFF_K, MR_SCRATCH);
}

}  // namespace

cudaError_t launch_decode_mr(const DecodeArgs& a, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDecodeDevices) return cudaErrorInvalidDevice;
  static std::once_flag once[kMaxDecodeDevices];
  static cudaError_t setup_err[kMaxDecodeDevices];
  std::call_once(once[dev], [&] {
    setup_err[dev] = cudaFuncSetAttribute(decode_mr_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, MR_SMEM);
  });
  if (setup_err[dev] != cudaSuccess) return setup_err[dev];
  DecodeArgs c = a;
  c.pps = 1;  // one partial per key slice
  c.ptrans = 0;
  c.coop = 0;
  return launch_k(decode_mr_kernel, dim3(a.num_kv_heads, a.batch, a.num_splits), dim3(MR_THREADS), MR_SMEM, s, c);
}

}  // namespace ftkv
