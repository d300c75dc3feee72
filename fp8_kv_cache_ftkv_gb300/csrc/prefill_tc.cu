// prefill_tc.cu -- prefill (extend) attention on the sm_100-family tensor cores (tcgen05 + TMA + TMEM).
//
// What it computes (FreeToken PR #853, "What changes"): chunk query t attends to every key of the
// reconstructed BF16 prefix and to chunk keys 0..t; the current chunk's K/V stay BF16.
//
// One CTA = 128 query rows of one query head (grid: query tiles x heads, heaviest tiles first).
// Key tiles of 128 keys come first from the prefix workspace, then from the chunk (causal tiles only).
//   warp 0      : TMEM allocation; lane 0 issues the TMA loads of Q and of the K tiles into a 3-stage K ring
//   warp 6      : lane 0 issues the TMA loads of the V tiles into a 3-stage V ring.  A K stage is refilled as
//                 soon as its QK product is done, a V stage once its PV product is done (one shared K+V
//                 stage waited for the PV product, which exposed the tile load latency in every tile)
//   warp 1      : lane 0 issues tcgen05.mma: S_j = Q K_j^T into one of two TMEM S buffers, then
//                 O += P_{j-1} V_{j-1} into the TMEM O accumulator, P read from TMEM (so QK of the next
//                 tile overlaps the softmax of the current one)
//   warps 2..5  : softmax, one query row per thread (= one TMEM lane): reads S_j from TMEM, keeps the
//                 running max/sum in registers (the max on raw scores, the scale folded into the exponent's
//                 FMA; packed f32x2 arithmetic and three-input max), writes P_j (BF16 pairs) into one of
//                 two TMEM P buffers (its own lane), and rescales the O row in TMEM only when the running
//                 max grew by more than 8 (log2 units), so the O correction is rare.  Keeping P in TMEM
//                 leaves the shared memory to the Q tile and the two 3-stage rings
// Operands: Q, K are K-major with the 128-byte swizzle; P is the TMEM A operand of the PV product; V is
// MN-major (keys x d, d contiguous) with the 128-byte swizzle, read directly by the tensor core.  Every mbarrier wait is bounded in time; on
// expiry the CTA records an error flag, drains its outstanding operations and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "ftkv_device.cuh"
#include "ftkv_internal.h"

namespace ftkv {
namespace {

constexpr int BM = 128;                    // query rows per CTA (MMA M)
constexpr int BN = 128;                    // keys per tile (MMA N of QK, MMA K of PV)
constexpr uint32_t BOX_BYTES = 128 * 128;  // one TMA box: 128 rows x 64 BF16 (128 B)
constexpr uint32_t TILE_BYTES = 2 * BOX_BYTES;  // 128 rows x 128 BF16
// shared-memory layout (offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_Q = 0;
constexpr int NS = 3;                                            // stages of the K ring and of the V ring
constexpr uint32_t OFF_K = OFF_Q + TILE_BYTES;                   // K stage s at +s*TILE
constexpr uint32_t OFF_V = OFF_K + NS * TILE_BYTES;              // V stage s at +s*TILE
constexpr uint32_t OFF_BAR = OFF_V + NS * TILE_BYTES;
constexpr int NBAR = 22;
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;              // TMEM base address, abort flag
constexpr uint32_t SMEM_USED = OFF_MISC + 16;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;              // slack for the 1024-byte alignment
static_assert(SMEM_ALLOC <= 232448, "prefill_tc shared memory");

// barrier indices
constexpr int B_QFULL = 0, B_FULL0 = 1, B_EMPTY0 = 4, B_FULLV0 = 7, B_EMPTYV0 = 10,  // K ring, V ring (NS each)
              B_SFULL0 = 13, B_SFREE0 = 15, B_PFULL0 = 17, B_ODONE = 19, B_OFINAL = 20, B_DRAIN = 21;

constexpr uint32_t TMEM_COLS = 512;        // S0 [0,128) S1 [128,256) O [256,384) P0 [384,448) P1 [448,512)
constexpr uint32_t TMEM_O = 256;
constexpr uint32_t TMEM_P = 384;           // P buffer b: 128 keys as 64 columns of packed BF16 pairs
constexpr unsigned long long WAIT_LIMIT_NS = 4000000000ull;   // 4 s

struct TcArgs {
  int num_q_heads;
  int group;
  int chunk_len;
  int prefix_len;
  int n_q_tiles;
  float qk_scale_log2;
  uint16_t* out;
  int* err;
  // two-heads-per-CTA kernel: key tiles per head pair (all its query tiles), and stream-K scheduling
  long long sk_wpair;
  long long sk_units;   // sk_wpair x head pairs
  int sk_ctas;          // persistent CTAs (0: one CTA per item)
  float* sk_part;       // [sk_ctas + 1 boundaries][2 pieces][piece floats]
  int* sk_ticket;       // [sk_ctas + 1 boundaries][4 softmax warps], zero between calls
};

// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity.  Returns false (and raises the CTA abort flag and
// the device error word) if it does not complete within WAIT_LIMIT_NS or another thread aborted.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > WAIT_LIMIT_NS) {
      *abort_flag = 1;
      flag_error(err, kDevErrTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// tcgen05 shared-memory matrix descriptor: start, leading / stride byte offsets, 128-byte swizzle.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;  // swizzle: 128 bytes
  return d;
}

// Instruction descriptor, kind::f16: FP32 accumulate, BF16 A and B, M = 128, N = 128.
__host__ __device__ constexpr uint32_t idesc_bf16(bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((128u >> 3) << 17) |
         ((128u >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D += A B with A read from tensor memory (128 lanes = rows, 8 columns = 16 BF16 of K) and B from shared memory
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
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
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]),
      "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]),
      "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]),
      "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// K-major SW128 tile of 128 rows x 128 BF16 (two 64-column boxes of 16 KB): descriptor of k-step kk
// (16 columns) for the MMA.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) {
  return sw128_desc(tile + (kk >> 2) * BOX_BYTES + (kk & 3) * 32, 16, 1024);
}
// MN-major SW128 V tile (128 keys x 128 d, d contiguous; two 64-d boxes): k-step kk covers keys
// 16kk..16kk+15 (two 8-row swizzle atoms); the two 64-d atoms are BOX_BYTES apart.
__device__ __forceinline__ uint64_t vtile_desc(uint32_t tile, int kk) {
  return sw128_desc(tile + kk * 2048, BOX_BYTES, 1024);
}

// Packed FP32 pairs (one instruction for two lanes of work) and the three-input maximum.
__device__ __forceinline__ float2 ffma2(float2 x, float2 y, float2 z) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<unsigned long long*>(&x)), "l"(*reinterpret_cast<unsigned long long*>(&y)),
        "l"(*reinterpret_cast<unsigned long long*>(&z)));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float2 fadd2(float2 x, float2 y) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<unsigned long long*>(&x)), "l"(*reinterpret_cast<unsigned long long*>(&y)));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float fmax3(float x, float y, float z) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(x), "f"(y), "f"(z));
  return d;
}

// Row maximum of 128 scores as four independent chains (a single chain is 64 dependent fmax3 deep).
__device__ __forceinline__ float row_max(const float (&s)[BN]) {
  float m0 = fmaxf(s[0], s[1]), m1 = fmaxf(s[2], s[3]), m2 = fmaxf(s[4], s[5]), m3 = fmaxf(s[6], s[7]);
#pragma unroll
  for (int c = 8; c < BN; c += 8) {
    m0 = fmax3(m0, s[c], s[c + 1]);
    m1 = fmax3(m1, s[c + 2], s[c + 3]);
    m2 = fmax3(m2, s[c + 4], s[c + 5]);
    m3 = fmax3(m3, s[c + 6], s[c + 7]);
  }
  return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
}

constexpr int NTHREADS = 224;  // K producer, MMA issuer, 4 softmax warps, V producer

__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tkc,
                      const __grid_constant__ CUtensorMap tvc, const __grid_constant__ CUtensorMap twk,
                      const __grid_constant__ CUtensorMap twv, const TcArgs a) {
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + OFF_MISC + 4);
  const uint32_t tmem_holder = base + OFF_MISC;
  auto bar = [&](int i) { return base + OFF_BAR + 8u * i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = a.n_q_tiles - 1 - static_cast<int>(blockIdx.x);  // heaviest (latest) query tiles first
  const int hq = blockIdx.y;
  const int hk = hq / a.group;
  const int t0 = qt * BM;
  const int nPT = (a.prefix_len + BN - 1) / BN;
  const int last_q = (t0 + BM - 1 < a.chunk_len - 1) ? t0 + BM - 1 : a.chunk_len - 1;
  const int nCT = last_q / BN + 1;
  const int T = nPT + nCT;

  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 1);
    for (int s = 0; s < NS; s++) {
      mbar_init(bar(B_FULL0 + s), 1);
      mbar_init(bar(B_EMPTY0 + s), 1);
      mbar_init(bar(B_FULLV0 + s), 1);
      mbar_init(bar(B_EMPTYV0 + s), 1);
    }
    for (int s = 0; s < 2; s++) {
      mbar_init(bar(B_SFULL0 + s), 1);
      mbar_init(bar(B_SFREE0 + s), 128);
      mbar_init(bar(B_PFULL0 + s), 128);
    }
    mbar_init(bar(B_ODONE), 1);
    mbar_init(bar(B_OFINAL), 1);
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tmem_holder),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + OFF_MISC);

  if (warp == 0 || warp == 6) {
    if (lane == 0) {
      // ---------------- TMA producers: warp 0 Q and the K tiles, warp 6 the V tiles ----------------
      const bool is_k = warp == 0;
      if (is_k) {
        mbar_expect_tx(bar(B_QFULL), TILE_BYTES);
        tma_load_3d(base + OFF_Q, &tq, bar(B_QFULL), 0, hq, t0);
        tma_load_3d(base + OFF_Q + BOX_BYTES, &tq, bar(B_QFULL), 64, hq, t0);
      }
      const int FULL = is_k ? B_FULL0 : B_FULLV0, EMPTY = is_k ? B_EMPTY0 : B_EMPTYV0;
      int issued = 0;
      for (int j = 0; j < T; j++) {
        const int s = j % NS, use = j / NS;  // stage, and how often it was filled before
        if (use >= 1 && !mbar_wait(bar(EMPTY + s), (use - 1) & 1, abort_flag, a.err)) break;
        const bool pre = j < nPT;
        const CUtensorMap* m = is_k ? (pre ? &twk : &tkc) : (pre ? &twv : &tvc);
        const int row = pre ? j * BN : (j - nPT) * BN;
        const uint32_t d = base + (is_k ? OFF_K : OFF_V) + s * TILE_BYTES;
        mbar_expect_tx(bar(FULL + s), TILE_BYTES);
        tma_load_3d(d, m, bar(FULL + s), 0, hk, row);
        tma_load_3d(d + BOX_BYTES, m, bar(FULL + s), 64, hk, row);
        issued = j + 1;
      }
      // drain: every issued load must land before the CTA may exit
      if (is_k) mbar_wait(bar(B_QFULL), 0, abort_flag, a.err);
      for (int j = (issued > NS ? issued - NS : 0); j < issued; j++) mbar_wait(bar(FULL + j % NS), (j / NS) & 1, abort_flag, a.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t IDESC_QK = idesc_bf16(false);
      constexpr uint32_t IDESC_PV = idesc_bf16(true);
      bool ok = mbar_wait(bar(B_QFULL), 0, abort_flag, a.err);
      auto issue_pv = [&](int i) -> bool {
        const int b = i & 1, sv = i % NS;
        if (!mbar_wait(bar(B_PFULL0 + b), (i >> 1) & 1, abort_flag, a.err)) return false;
        if (!mbar_wait(bar(B_FULLV0 + sv), (i / NS) & 1, abort_flag, a.err)) return false;
        tc_fence_after();
        const uint32_t vt = base + OFF_V + sv * TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < 8; kk++)
          umma_bf16_ta(tmem + TMEM_O, tmem + TMEM_P + b * 64 + kk * 8, vtile_desc(vt, kk), IDESC_PV,
                       (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(bar(B_EMPTYV0 + sv));
        umma_commit(bar(B_ODONE));
        return true;
      };
      for (int j = 0; ok && j < T; j++) {
        const int s = j & 1;
        if (!mbar_wait(bar(B_FULL0 + j % NS), (j / NS) & 1, abort_flag, a.err)) { ok = false; break; }
        if (j >= 2 && !mbar_wait(bar(B_SFREE0 + s), ((j >> 1) - 1) & 1, abort_flag, a.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t kt = base + OFF_K + (j % NS) * TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < 8; kk++)
          umma_bf16(tmem + s * 128, kmajor_desc(base + OFF_Q, kk), kmajor_desc(kt, kk), IDESC_QK, kk > 0 ? 1u : 0u);
        umma_commit(bar(B_SFULL0 + s));
        umma_commit(bar(B_EMPTY0 + j % NS));  // K tile j is consumed once its QK product is done
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok && issue_pv(T - 1)) umma_commit(bar(B_OFINAL));
      // drain every MMA issued by this thread before TMEM is released
      umma_commit(bar(B_DRAIN));
      mbar_wait(bar(B_DRAIN), 0, abort_flag, a.err);
    }
  } else {  // warps 2..5
    // ---------------- softmax: one query row per thread ----------------
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int t = t0 + row;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float m_used = -INFINITY, lsum = 0.0f;
    bool ok = true;
    float s[BN];
    for (int j = 0; j < T && ok; j++) {
      const int b = j & 1;
      // wait results are made warp-uniform before any warp-collective tcgen05 access
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_SFULL0 + b), (j >> 1) & 1, abort_flag, a.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 4; c++) tmem_ld32(lane_base + b * 128 + c * 32, s + c * 32);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(bar(B_SFREE0 + b));

      const bool pre = j < nPT;
      const int kbase = pre ? j * BN : (j - nPT) * BN;
      const int lim = pre ? a.prefix_len - kbase : (t + 1 - kbase);  // columns < lim are visible
      // Tile maximum on the raw scores (the scale is positive: same order), masking only boundary tiles;
      // the scale is applied once, to the maximum, and folded into the exponent's FMA below.
      if (lim < BN) {
#pragma unroll
        for (int c = 0; c < BN; c++) s[c] = (c < lim) ? s[c] : -INFINITY;
      }
      const float mraw = row_max(s);
      const float mt = mraw * a.qk_scale_log2;
      const float m_new = fmaxf(m_used, mt);
      const bool need = (m_used != -INFINITY) && (m_new > m_used + 8.0f);
      if (m_used == -INFINITY) m_used = m_new;
      if (__any_sync(0xffffffffu, need)) {
        const float f = need ? fast_exp2(m_used - m_new) : 1.0f;
        if (need) {
          lsum *= f;
          m_used = m_new;
        }
        if (j >= 1) {  // O holds PV_0..PV_{j-1}: wait for the last of them, then scale the row in place
          if (!__all_sync(0xffffffffu, mbar_wait(bar(B_ODONE), (j - 1) & 1, abort_flag, a.err))) {
            ok = false;
            break;
          }
          tc_fence_after();
          float o[32];
#pragma unroll
          for (int c = 0; c < 4; c++) {
            tmem_ld32(lane_base + TMEM_O + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; e++) o[e] *= f;
            tmem_st32(lane_base + TMEM_O + c * 32, o);
          }
          tmem_st_wait();
        }
      }
      const float sub = (m_used == -INFINITY) ? 0.0f : m_used;
      // P row (BF16 pairs) into TMEM P buffer b, this thread's lane, columns 0..63; p = 2^(s scale - sub),
      // exponents and sums in pairs
      const float2 scale2 = make_float2(a.qk_scale_log2, a.qk_scale_log2), nsub2 = make_float2(-sub, -sub);
      float2 ps2[4] = {};  // four independent partial sums
#pragma unroll
      for (int half = 0; half < 2; half++) {
        float w[32];  // 32 packed BF16 pairs, as raw 32-bit words
#pragma unroll
        for (int e = 0; e < 32; e++) {
          const int c = half * 64 + 2 * e;
          const float2 arg = ffma2(make_float2(s[c], s[c + 1]), scale2, nsub2);
          const float2 pp = make_float2(fast_exp2(arg.x), fast_exp2(arg.y));
          ps2[e & 3] = fadd2(ps2[e & 3], pp);
          w[e] = __uint_as_float(float2_to_bf16x2(pp.x, pp.y));
        }
        tmem_st32(lane_base + TMEM_P + b * 64 + half * 32, w);
      }
      lsum += ((ps2[0].x + ps2[1].x) + (ps2[2].x + ps2[3].x)) + ((ps2[0].y + ps2[1].y) + (ps2[2].y + ps2[3].y));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL0 + b));
    }
    // ---- epilogue: O / l -> BF16 ----
    if (__all_sync(0xffffffffu, ok && mbar_wait(bar(B_OFINAL), 0, abort_flag, a.err))) {
      tc_fence_after();
      const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
      uint16_t* dst = a.out + (static_cast<int64_t>(t) * a.num_q_heads + hq) * kHeadDim;
#pragma unroll
      for (int c = 0; c < 4; c++) {
        float o[32];
        tmem_ld32(lane_base + TMEM_O + c * 32, o);
        tmem_ld_wait();
        if (t < a.chunk_len) {
#pragma unroll
          for (int q = 0; q < 4; q++) {
            uint4 v;
            v.x = float2_to_bf16x2(o[q * 8 + 0] * inv, o[q * 8 + 1] * inv);
            v.y = float2_to_bf16x2(o[q * 8 + 2] * inv, o[q * 8 + 3] * inv);
            v.z = float2_to_bf16x2(o[q * 8 + 4] * inv, o[q * 8 + 5] * inv);
            v.w = float2_to_bf16x2(o[q * 8 + 6] * inv, o[q * 8 + 7] * inv);
            *reinterpret_cast<uint4*>(dst + c * 32 + q * 8) = v;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// ---------------------------------------------------------------------------------------------
// Two query heads per CTA (even GQA groups).  Query heads 2y and 2y+1 share a KV head, so one K/V stream
// feeds both: each K/V tile is fetched once for two heads, which halves the tile bytes per unit of work
// (what bounds the one-head kernel).  The softmax warpgroup alternates between the heads, and each
// head's tensor-core work overlaps the other head's softmax.  TMEM: S_h at columns [128h, 128h + 128),
// P_h written over the first 64 of them (BF16 pairs) once S_h is in registers; O_h at [256 + 128h, ...).
// The QK product of the next tile into S_h is issued after PV_h, so the in-order tensor pipe never
// overwrites a P it has not read.  Issue order: QK_0(0) QK_1(0) | PV_0(j) QK_0(j+1) PV_1(j) QK_1(j+1) ...
//
// Work items are (head pair y, query tile qt), T = nPT + qt + 1 key tiles each.  Either one CTA per item
// (sk_ctas == 0), or stream-K: the items' tiles, laid end to end (pair-major, qt ascending), are cut into
// sk_ctas equal ranges, one per persistent CTA, so every SM gets the same number of tiles whatever the
// mix of item sizes.  A CTA runs the segments (item, tile range) of its range in order.  An item cut by a
// range boundary has two pieces, in CTAs c and c+1: each writes its unnormalised O, its running max and
// its sum to the boundary's slot and takes a ticket (one per softmax warp and its 32 rows); the second
// to arrive merges the two
// (o = (2^(m0-m) O0 + 2^(m1-m) O1) / (2^(m0-m) l0 + 2^(m1-m) l1), m = max) and resets the ticket.
// Ranges are at least as long as the largest item, so no item has more than two pieces.
namespace tc2 {
constexpr int NSK = 3, NSV = 2;                                   // K and V ring stages
constexpr uint32_t OFF_Q = 0;                                     // head h at +h*TILE
constexpr uint32_t OFF_K = 2 * TILE_BYTES;                        // K stage s at +s*TILE
constexpr uint32_t OFF_V = OFF_K + NSK * TILE_BYTES;              // V stage s at +s*TILE
constexpr uint32_t OFF_BAR = OFF_V + NSV * TILE_BYTES;
constexpr int B_QFULL = 0, B_FULL0 = 1, B_EMPTY0 = 4, B_FULLV0 = 7, B_EMPTYV0 = 9, B_SFULL0 = 11, B_PFULL0 = 13,
              B_ODONE0 = 15, B_OFREE0 = 17, B_QEMPTY = 19, B_DRAIN = 20, NBAR = 21;
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;                 // TMEM base address, abort flag
constexpr uint32_t SMEM_ALLOC = OFF_MISC + 16 + 1024;             // + slack for the 1024-byte alignment
static_assert(SMEM_ALLOC <= 232448, "prefill_tc2 shared memory");
// One piece of a cut item: O [head][d/4][row][4] FP32 (a warp's rows read and write 512 contiguous bytes),
// then m [head][row] and l [head][row].
constexpr int PIECE_FLOATS = 2 * BM * kHeadDim + 4 * BM;
}  // namespace tc2

// A segment: head pair p, query tile qt, key tiles [ja, jb) of the item's T.
struct Seg {
  int p, qt, ja, jb, T;
};

// The next segment of the unit range [u, u1), advancing u; false when the range is used up.
__device__ __forceinline__ bool next_segment(long long& u, long long u1, const TcArgs& a, int nPT, Seg& sg) {
  if (u >= u1) return false;
  sg.p = static_cast<int>(u / a.sk_wpair);
  const long long rem = u - static_cast<long long>(sg.p) * a.sk_wpair;
  int qt = 0;
  long long base = 0;
  while (qt + 1 < a.n_q_tiles && base + nPT + qt + 1 <= rem) {
    base += nPT + qt + 1;
    qt++;
  }
  sg.qt = qt;
  sg.T = nPT + qt + 1;
  sg.ja = static_cast<int>(rem - base);
  const long long left = u1 - u;
  sg.jb = (sg.ja + left < sg.T) ? sg.ja + static_cast<int>(left) : sg.T;
  u += sg.jb - sg.ja;
  return true;
}

__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_tc2_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tkc,
                       const __grid_constant__ CUtensorMap tvc, const __grid_constant__ CUtensorMap twk,
                       const __grid_constant__ CUtensorMap twv, const TcArgs a) {
  using tc2::NSK, tc2::NSV, tc2::OFF_Q, tc2::OFF_K, tc2::OFF_V, tc2::OFF_BAR, tc2::OFF_MISC, tc2::PIECE_FLOATS;
  using tc2::B_QFULL, tc2::B_FULL0, tc2::B_EMPTY0, tc2::B_FULLV0, tc2::B_EMPTYV0, tc2::B_SFULL0, tc2::B_PFULL0,
      tc2::B_ODONE0, tc2::B_OFREE0, tc2::B_QEMPTY, tc2::B_DRAIN;
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + OFF_MISC + 4);
  const uint32_t tmem_holder = base + OFF_MISC;
  auto bar = [&](int i) { return base + OFF_BAR + 8u * i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nPT = (a.prefix_len + BN - 1) / BN;
  // this CTA's unit range: stream-K, or the one item of (blockIdx.x, blockIdx.y) (heaviest first)
  long long u_begin, u_end;
  if (a.sk_ctas > 0) {
    u_begin = static_cast<long long>(blockIdx.x) * a.sk_units / a.sk_ctas;
    u_end = static_cast<long long>(blockIdx.x + 1) * a.sk_units / a.sk_ctas;
  } else {
    const int qt = a.n_q_tiles - 1 - static_cast<int>(blockIdx.x);
    u_begin = static_cast<long long>(blockIdx.y) * a.sk_wpair + static_cast<long long>(qt) * nPT +
              static_cast<long long>(qt) * (qt + 1) / 2;
    u_end = u_begin + nPT + qt + 1;
  }

  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QEMPTY), 1);
    for (int s = 0; s < NSK; s++) {
      mbar_init(bar(B_FULL0 + s), 1);
      mbar_init(bar(B_EMPTY0 + s), 1);
    }
    for (int s = 0; s < NSV; s++) {
      mbar_init(bar(B_FULLV0 + s), 1);
      mbar_init(bar(B_EMPTYV0 + s), 1);
    }
    for (int h = 0; h < 2; h++) {
      mbar_init(bar(B_SFULL0 + h), 1);
      mbar_init(bar(B_PFULL0 + h), 128);
      mbar_init(bar(B_ODONE0 + h), 1);
      mbar_init(bar(B_OFREE0 + h), 128);
    }
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tmem_holder),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + OFF_MISC);

  if (warp == 0 || warp == 6) {
    if (lane == 0) {
      // ---------------- TMA producers: warp 0 the two Q tiles and the K tiles, warp 6 the V tiles ----------------
      const bool is_k = warp == 0;
      const int FULL = is_k ? B_FULL0 : B_FULLV0, EMPTY = is_k ? B_EMPTY0 : B_EMPTYV0;
      const int NS = is_k ? NSK : NSV;
      int issued = 0, nseg = 0;  // tiles issued (all segments), segments started
      bool ok = true;
      long long u = u_begin;
      Seg sg;
      while (ok && next_segment(u, u_end, a, nPT, sg)) {
        const int hq0 = 2 * sg.p, hk = hq0 / a.group, t0 = sg.qt * BM;
        if (is_k) {  // the segment's Q tiles, once the previous segment's QK products are done with Q
          if (nseg >= 1 && !mbar_wait(bar(B_QEMPTY), (nseg - 1) & 1, abort_flag, a.err)) break;
          mbar_expect_tx(bar(B_QFULL), 2 * TILE_BYTES);
          for (int h = 0; h < 2; h++) {
            tma_load_3d(base + OFF_Q + h * TILE_BYTES, &tq, bar(B_QFULL), 0, hq0 + h, t0);
            tma_load_3d(base + OFF_Q + h * TILE_BYTES + BOX_BYTES, &tq, bar(B_QFULL), 64, hq0 + h, t0);
          }
        }
        nseg++;
        for (int j = sg.ja; j < sg.jb; j++) {
          const int s = issued % NS, use = issued / NS;  // stage, and how often it was filled before
          if (use >= 1 && !mbar_wait(bar(EMPTY + s), (use - 1) & 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          const bool pre = j < nPT;
          const CUtensorMap* m = is_k ? (pre ? &twk : &tkc) : (pre ? &twv : &tvc);
          const int row = pre ? j * BN : (j - nPT) * BN;
          const uint32_t d = base + (is_k ? OFF_K : OFF_V) + s * TILE_BYTES;
          mbar_expect_tx(bar(FULL + s), TILE_BYTES);
          tma_load_3d(d, m, bar(FULL + s), 0, hk, row);
          tma_load_3d(d + BOX_BYTES, m, bar(FULL + s), 64, hk, row);
          issued++;
        }
      }
      // drain: every issued load must land before the CTA may exit
      if (is_k && nseg >= 1) mbar_wait(bar(B_QFULL), (nseg - 1) & 1, abort_flag, a.err);
      for (int j = (issued > NS ? issued - NS : 0); j < issued; j++) mbar_wait(bar(FULL + j % NS), (j / NS) & 1, abort_flag, a.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t IDESC_QK = idesc_bf16(false);
      constexpr uint32_t IDESC_PV = idesc_bf16(true);
      bool ok = true;
      int nseg = 0, g0 = 0;  // segments done, global index of the segment's first tile
      long long u = u_begin;
      Seg sg;
      auto qk = [&](int g, int h) {  // S_h = Q_h K_g^T
        const uint32_t kt = base + OFF_K + (g % NSK) * TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < 8; kk++)
          umma_bf16(tmem + h * 128, kmajor_desc(base + OFF_Q + h * TILE_BYTES, kk), kmajor_desc(kt, kk), IDESC_QK,
                    kk > 0 ? 1u : 0u);
        umma_commit(bar(B_SFULL0 + h));
      };
      auto wait_k = [&](int g) -> bool {
        if (!mbar_wait(bar(B_FULL0 + g % NSK), (g / NSK) & 1, abort_flag, a.err)) return false;
        tc_fence_after();
        return true;
      };
      while (ok && next_segment(u, u_end, a, nPT, sg)) {
        const int n = sg.jb - sg.ja, glast = g0 + n - 1;
        if (!mbar_wait(bar(B_QFULL), nseg & 1, abort_flag, a.err) || !wait_k(g0)) {
          ok = false;
          break;
        }
        qk(g0, 0);
        qk(g0, 1);
        umma_commit(bar(B_EMPTY0 + g0 % NSK));
        if (n == 1) umma_commit(bar(B_QEMPTY));
        auto pv = [&](int g, int h) -> bool {  // O_h += P_h V_g, P_h from TMEM
          if (!mbar_wait(bar(B_PFULL0 + h), g & 1, abort_flag, a.err)) return false;
          if (h == 0 && !mbar_wait(bar(B_FULLV0 + g % NSV), (g / NSV) & 1, abort_flag, a.err)) return false;
          // the first PV of a segment overwrites O_h: the previous segment's epilogue must have read it
          if (g == g0 && nseg >= 1 && !mbar_wait(bar(B_OFREE0 + h), (nseg - 1) & 1, abort_flag, a.err)) return false;
          tc_fence_after();
          const uint32_t vt = base + OFF_V + (g % NSV) * TILE_BYTES;
#pragma unroll
          for (int kk = 0; kk < 8; kk++)
            umma_bf16_ta(tmem + TMEM_O + h * 128, tmem + h * 128 + kk * 8, vtile_desc(vt, kk), IDESC_PV,
                         (g > g0 || kk > 0) ? 1u : 0u);
          umma_commit(bar(B_ODONE0 + h));
          if (h == 1) umma_commit(bar(B_EMPTYV0 + g % NSV));  // both PV products of tile g read its V stage
          return true;
        };
        for (int g = g0; g <= glast; g++) {
          if (!pv(g, 0)) { ok = false; break; }
          const bool more = g < glast;
          if (more) {
            if (!wait_k(g + 1)) { ok = false; break; }
            qk(g + 1, 0);
          }
          if (!pv(g, 1)) { ok = false; break; }
          if (more) {
            qk(g + 1, 1);
            umma_commit(bar(B_EMPTY0 + (g + 1) % NSK));  // both QK products of tile g+1 read its K stage
            if (g + 1 == glast) umma_commit(bar(B_QEMPTY));  // the segment's last QK products read Q
          }
        }
        nseg++;
        g0 += n;
      }
      // drain every MMA issued by this thread before TMEM is released
      umma_commit(bar(B_DRAIN));
      mbar_wait(bar(B_DRAIN), 0, abort_flag, a.err);
    }
  } else {  // warps 2..5
    // ---------------- softmax: one query row per thread, the two heads in turn ----------------
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    bool ok = true;
    float s[BN];
    int g0 = 0;
    long long u = u_begin;
    Seg sg;
    while (ok && next_segment(u, u_end, a, nPT, sg)) {
      const int hq0 = 2 * sg.p, t = sg.qt * BM + row;
      const int n = sg.jb - sg.ja, glast = g0 + n - 1;
      float m_used[2] = {-INFINITY, -INFINITY}, lsum[2] = {0.0f, 0.0f};
      for (int j = sg.ja; j < sg.jb && ok; j++) {
        const int g = g0 + (j - sg.ja);
        const bool pre = j < nPT;
        const int kbase = pre ? j * BN : (j - nPT) * BN;
        const int lim = pre ? a.prefix_len - kbase : (t + 1 - kbase);  // columns < lim are visible
#pragma unroll
        for (int h = 0; h < 2; h++) {
          // wait results are made warp-uniform before any warp-collective tcgen05 access
          if (!__all_sync(0xffffffffu, mbar_wait(bar(B_SFULL0 + h), g & 1, abort_flag, a.err))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 4; c++) tmem_ld32(lane_base + h * 128 + c * 32, s + c * 32);
          tmem_ld_wait();
          if (lim < BN) {
#pragma unroll
            for (int c = 0; c < BN; c++) s[c] = (c < lim) ? s[c] : -INFINITY;
          }
          const float mraw = row_max(s);
          const float mt = mraw * a.qk_scale_log2;
          const float m_new = fmaxf(m_used[h], mt);
          const bool need = (m_used[h] != -INFINITY) && (m_new > m_used[h] + 8.0f);
          if (m_used[h] == -INFINITY) m_used[h] = m_new;
          if (__any_sync(0xffffffffu, need)) {
            const float f = need ? fast_exp2(m_used[h] - m_new) : 1.0f;
            if (need) {
              lsum[h] *= f;
              m_used[h] = m_new;
            }
            if (g > g0) {  // O_h holds PV_h of the segment's earlier tiles: wait for the last, scale in place
              if (!__all_sync(0xffffffffu, mbar_wait(bar(B_ODONE0 + h), (g - 1) & 1, abort_flag, a.err))) {
                ok = false;
                break;
              }
              tc_fence_after();
              float o[32];
#pragma unroll
              for (int c = 0; c < 4; c++) {
                tmem_ld32(lane_base + TMEM_O + h * 128 + c * 32, o);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; e++) o[e] *= f;
                tmem_st32(lane_base + TMEM_O + h * 128 + c * 32, o);
              }
              tmem_st_wait();
            }
          }
          const float sub = (m_used[h] == -INFINITY) ? 0.0f : m_used[h];
          // P_h row (BF16 pairs) over the first 64 columns of S_h; p = 2^(s scale - sub), in pairs
          const float2 scale2 = make_float2(a.qk_scale_log2, a.qk_scale_log2), nsub2 = make_float2(-sub, -sub);
          float2 ps2[4] = {};  // four independent partial sums
#pragma unroll
          for (int half = 0; half < 2; half++) {
            float w[32];  // 32 packed BF16 pairs, as raw 32-bit words
#pragma unroll
            for (int e = 0; e < 32; e++) {
              const int c = half * 64 + 2 * e;
              const float2 arg = ffma2(make_float2(s[c], s[c + 1]), scale2, nsub2);
              const float2 pp = make_float2(fast_exp2(arg.x), fast_exp2(arg.y));
              ps2[e & 3] = fadd2(ps2[e & 3], pp);
              w[e] = __uint_as_float(float2_to_bf16x2(pp.x, pp.y));
            }
            tmem_st32(lane_base + h * 128 + half * 32, w);
          }
          lsum[h] += ((ps2[0].x + ps2[1].x) + (ps2[2].x + ps2[3].x)) + ((ps2[0].y + ps2[1].y) + (ps2[2].y + ps2[3].y));
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(B_PFULL0 + h));
        }
      }
      if (!ok) break;
      // ---- segment epilogue: a whole item writes O_h / l_h as BF16; a piece of a cut item writes its
      // partial (O_h, m_h, l_h) to the boundary's slot, and the second piece to arrive merges ----
      const bool whole = sg.ja == 0 && sg.jb == sg.T;
      const int bnd = (sg.ja > 0) ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x) + 1;  // boundary
      float* piece = whole ? nullptr
                           : a.sk_part + (static_cast<long long>(bnd) * 2 + (sg.ja > 0 ? 1 : 0)) * PIECE_FLOATS;
#pragma unroll
      for (int h = 0; h < 2; h++) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_ODONE0 + h), glast & 1, abort_flag, a.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float inv = lsum[h] > 0.0f ? 1.0f / lsum[h] : 0.0f;
        uint16_t* dst = a.out + (static_cast<int64_t>(t) * a.num_q_heads + hq0 + h) * kHeadDim;
#pragma unroll
        for (int c = 0; c < 4; c++) {
          float o[32];
          tmem_ld32(lane_base + TMEM_O + h * 128 + c * 32, o);
          tmem_ld_wait();
          if (whole) {
            if (t < a.chunk_len) {
#pragma unroll
              for (int q = 0; q < 4; q++) {
                uint4 v;
                v.x = float2_to_bf16x2(o[q * 8 + 0] * inv, o[q * 8 + 1] * inv);
                v.y = float2_to_bf16x2(o[q * 8 + 2] * inv, o[q * 8 + 3] * inv);
                v.z = float2_to_bf16x2(o[q * 8 + 4] * inv, o[q * 8 + 5] * inv);
                v.w = float2_to_bf16x2(o[q * 8 + 6] * inv, o[q * 8 + 7] * inv);
                *reinterpret_cast<uint4*>(dst + c * 32 + q * 8) = v;
              }
            }
          } else {
#pragma unroll
            for (int q = 0; q < 8; q++)
              *reinterpret_cast<float4*>(piece + ((h * 32 + c * 8 + q) * BM + row) * 4) =
                  make_float4(o[q * 4], o[q * 4 + 1], o[q * 4 + 2], o[q * 4 + 3]);
          }
        }
        if (!whole) {
          piece[2 * BM * kHeadDim + h * BM + row] = m_used[h];
          piece[2 * BM * kHeadDim + 2 * BM + h * BM + row] = lsum[h];
        }
        tc_fence_before();
        mbar_arrive(bar(B_OFREE0 + h));  // O_h is read: the next segment's first PV_h may overwrite it
      }
      if (!ok) break;
      if (!whole) {
        // one ticket per (boundary, warp): each softmax warp hands over its own 32 rows, so no barrier
        // joins the warps (a warp that gave up on a timeout cannot hold the others)
        __threadfence();
        __syncwarp();
        int prev = 0;
        if (lane == 0) {
          prev = atomicAdd(a.sk_ticket + bnd * 4 + quarter, 1);
          if (prev == 1) a.sk_ticket[bnd * 4 + quarter] = 0;  // both pieces are in: ready for the next call
        }
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == 1) {
          __threadfence();
          const float* p0 = a.sk_part + static_cast<long long>(bnd) * 2 * PIECE_FLOATS;
          const float* p1 = p0 + PIECE_FLOATS;
#pragma unroll 1
          for (int h = 0; h < 2; h++) {
            const float m0 = __ldcg(p0 + 2 * BM * kHeadDim + h * BM + row);
            const float m1 = __ldcg(p1 + 2 * BM * kHeadDim + h * BM + row);
            const float l0 = __ldcg(p0 + 2 * BM * kHeadDim + 2 * BM + h * BM + row);
            const float l1 = __ldcg(p1 + 2 * BM * kHeadDim + 2 * BM + h * BM + row);
            const float mm = fmaxf(m0, m1);
            const float f0 = (mm == -INFINITY) ? 0.0f : exp2f(m0 - mm);
            const float f1 = (mm == -INFINITY) ? 0.0f : exp2f(m1 - mm);
            const float L = l0 * f0 + l1 * f1;
            const float inv = L > 0.0f ? 1.0f / L : 0.0f;
            const float w0 = f0 * inv, w1 = f1 * inv;
            uint16_t* dst = a.out + (static_cast<int64_t>(t) * a.num_q_heads + hq0 + h) * kHeadDim;
#pragma unroll 4
            for (int c4 = 0; c4 < 32; c4 += 2) {
              const float4 x0 = __ldcg(reinterpret_cast<const float4*>(p0 + ((h * 32 + c4) * BM + row) * 4));
              const float4 y0 = __ldcg(reinterpret_cast<const float4*>(p0 + ((h * 32 + c4 + 1) * BM + row) * 4));
              const float4 x1 = __ldcg(reinterpret_cast<const float4*>(p1 + ((h * 32 + c4) * BM + row) * 4));
              const float4 y1 = __ldcg(reinterpret_cast<const float4*>(p1 + ((h * 32 + c4 + 1) * BM + row) * 4));
              if (t < a.chunk_len) {
                uint4 v;
                v.x = float2_to_bf16x2(x0.x * w0 + x1.x * w1, x0.y * w0 + x1.y * w1);
                v.y = float2_to_bf16x2(x0.z * w0 + x1.z * w1, x0.w * w0 + x1.w * w1);
                v.z = float2_to_bf16x2(y0.x * w0 + y1.x * w1, y0.y * w0 + y1.y * w1);
                v.w = float2_to_bf16x2(y0.z * w0 + y1.z * w1, y0.w * w0 + y1.w * w1);
                *reinterpret_cast<uint4*>(dst + c4 * 4) = v;
              }
            }
          }
        }
      }
      g0 += n;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// ---------------------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  // looked up once (thread-safe static initialisation); null if the driver lacks it
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// [rows][heads][128] BF16 as a 3-D tensor (d, head, row); box = 64 d x 1 head x 128 rows, 128-B swizzle.
bool make_map(CUtensorMap* m, const void* ptr, int heads, int64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {256, static_cast<cuuint64_t>(heads) * 256};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

// Stream-K workspace: tickets [max_ctas + 1][4] (rounded up to 256 bytes), then the pieces
// [max_ctas + 1][2][PIECE_FLOATS].
int64_t prefill_workspace_bytes(int max_ctas) {
  const int64_t n = max_ctas + 1;
  return (n * 4 * 4 + 255) / 256 * 256 + n * 2 * tc2::PIECE_FLOATS * 4;
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s) {
  // per-device set-up, once per device even with several host threads
  static std::once_flag once[kMaxDecodeDevices];
  static cudaError_t setup_err[kMaxDecodeDevices];
  int dev = 0;
  cudaError_t ge = cudaGetDevice(&dev);
  if (ge != cudaSuccess) return ge;
  if (dev < 0 || dev >= kMaxDecodeDevices) return cudaErrorInvalidDevice;
  std::call_once(once[dev], [&] {
    setup_err[dev] = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
    if (setup_err[dev] == cudaSuccess)
      setup_err[dev] =
          cudaFuncSetAttribute(prefill_tc2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tc2::SMEM_ALLOC);
  });
  if (setup_err[dev] != cudaSuccess) return setup_err[dev];
  CUtensorMap tq, tkc, tvc, twk, twv;
  if (!make_map(&tq, a.q, a.num_q_heads, a.chunk_len) || !make_map(&tkc, a.k_chunk, a.num_kv_heads, a.chunk_len) ||
      !make_map(&tvc, a.v_chunk, a.num_kv_heads, a.chunk_len))
    return cudaErrorInvalidValue;
  if (a.prefix_len > 0) {
    if (!make_map(&twk, a.ws_k, a.num_kv_heads, a.prefix_len) || !make_map(&twv, a.ws_v, a.num_kv_heads, a.prefix_len))
      return cudaErrorInvalidValue;
  } else {
    twk = tkc;
    twv = tvc;
  }
  TcArgs t{};
  t.num_q_heads = a.num_q_heads;
  t.group = a.num_q_heads / a.num_kv_heads;
  t.chunk_len = static_cast<int>(a.chunk_len);
  t.prefix_len = static_cast<int>(a.prefix_len);
  t.n_q_tiles = static_cast<int>((a.chunk_len + BM - 1) / BM);
  t.qk_scale_log2 = a.qk_scale_log2;
  t.out = a.out;
  t.err = a.err;
  if (t.group % 2 == 0) {  // query heads 2y and 2y+1 share a KV head: one CTA, one K/V stream for both
    const long long nPT = (a.prefix_len + BN - 1) / BN, nQT = t.n_q_tiles, pairs = a.num_q_heads / 2;
    t.sk_wpair = nQT * nPT + nQT * (nQT + 1) / 2;
    t.sk_units = pairs * t.sk_wpair;
    if (a.workspace) {
      // stream-K when there are more items than CTAs and every CTA's range holds a whole largest item
      // (so no item is cut twice); otherwise one CTA per item
      int cap = a.max_ctas;
      if (cap <= 0) {
        cudaError_t e = cudaDeviceGetAttribute(&cap, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
      }
      if (prefill_workspace_bytes(cap) > a.workspace_bytes) return cudaErrorInvalidValue;
      if (nQT * pairs > cap && t.sk_units / cap >= nPT + nQT) {
        t.sk_ctas = cap;
        t.sk_ticket = static_cast<int*>(a.workspace);
        t.sk_part = reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) +
                                             ((static_cast<int64_t>(cap + 1) * 4 * 4 + 255) / 256) * 256);
        return launch_k(prefill_tc2_kernel, dim3(cap), dim3(NTHREADS), tc2::SMEM_ALLOC, s, tq, tkc, tvc, twk, twv, t);
      }
    }
    dim3 grid(t.n_q_tiles, a.num_q_heads / 2);
    return launch_k(prefill_tc2_kernel, grid, dim3(NTHREADS), tc2::SMEM_ALLOC, s, tq, tkc, tvc, twk, twv, t);
  }
  dim3 grid(t.n_q_tiles, a.num_q_heads);
  return launch_k(prefill_tc_kernel, grid, dim3(NTHREADS), SMEM_ALLOC, s, tq, tkc, tvc, twk, twv, t);
}

}  // namespace ftkv
