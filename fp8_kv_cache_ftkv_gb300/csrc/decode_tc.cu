// decode_tc.cu -- single-row split-K decode attention on the tcgen05 tensor cores, fed by TMA gathers.
//
// What it computes (FreeToken PR #897, opening description and "Fresh R9700 stage-1 A/B"): for each
// query head i (KV head h = i / G) of a request with n cached keys,
//     o = sum_j softmax_j((q . k^_j) * sm_scale) v^_j,   k^_j = decode(codeK_j) scaleK_j, v^_j likewise,
// split over key slices whose partials (m, l, O) are merged by the slice that finishes last (the same
// partial format and merge as the warp-level kernel in decode.cu).  This kernel serves requests with
// one query row; the warp-level kernel serves the multi-row (MTP / speculative) case.
//
// CTA = (key slice, KV head, request), 16 warps, tiles of 128 keys, a 4-stage ring of 33 KB stages:
//   warps 0-3   producers.  They stage the slice's slot indices in shared memory (a double window of 2 x 2048;
//               the first window is requested before anything else, so its latency overlaps the set-up).
//               Per tile, each gather group of 4 keys gets one TMA tile::gather4 for its 4 K code rows
//               and one for its 4 V code rows (128-byte rows, 128-byte swizzle, box one row high); the
//               32 groups are spread over the producer warps, because a gather4 instruction issues its
//               lanes' operations one after another.  The scales are read with plain loads one tile
//               ahead and stored into the stage after the gathers are issued, before the warp's arrival
//               on the stage's mbarrier (expected bytes announced first, one arrival per warp).  Copies of 4-byte scales through cp.async,
//               or of the V rows through cp.async, slowed the gathers' issue severalfold when mixed with
//               them; TMA alone in flight issues at the rate of a pure-load kernel.  Padding keys past
//               the slice's end gather the head's row of slot 0 (in bounds) and get zero scales.
//   warp 4      TMEM owner; lane 0 issues the MMAs:
//                 S_i = K_i Qp^T    kind::f8f6f4, E4M3 x E4M3 -> FP32, M = 128 keys, N = 16 (8 query
//                                   heads x 2 exact E4M3 pieces of the BF16 query), K = 128 d; the
//                                   stored K codes are the A operand as they were gathered.
//                 D_i = Vh_i^T P'_i kind::f16, M = 128 d, N = 64 ((head half, block of 16 keys, head)
//                                   rows of P'), K = 128 keys; V is the MN-major A operand.
//               S and D are double-buffered in TMEM.
//   warps 5-12  softmax, two warps per TMEM lane quarter, each for 4 of the 8 query heads; a thread is one
//               key row of S and one d row of D.  Scores, exact per-tile maxima per head (redux.sync and
//               one shared-memory exchange), p = 2^(s - m), the value-weighted weight w = p scaleV, and
//               P' = w 2^-E in FP16 where 2^E is the power of two of the largest w of the key's 16-key
//               block for that head (every block keeps FP16's full range).  Then the fold
//               O = O alpha_i + sum_blocks D_i[block] 2^E[block] in FP32 registers.
//   warps 13-15 convert the V code tile to FP16 (packed hardware converter) in the MN-major SW128 layout,
//               writing zeros for padding keys.
// Every mbarrier wait is bounded by %globaltimer; on expiry the CTA flags FTKV_DEVERR_TIMEOUT, drains its
// loads and MMAs, releases TMEM and leaves its outputs unspecified.  The named barriers of the producer
// and softmax groups are crossed only with a group-uniform decision (a reduction or a vote at the
// barrier), so a timeout cannot strand a warp at a barrier the others skipped.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "decode_merge.cuh"
#include "ftkv_device.cuh"
#include "ftkv_internal.h"

namespace ftkv {
namespace {

constexpr int TK = 128;                                  // keys per tile
constexpr int NS = 4;                                    // stages of the load ring
constexpr int SLOT_CAP = 2048;                           // slot indices per window (two windows staged)
constexpr int NPROD = 4, NSOFT = 8, NCONV = 3;           // warps per role
constexpr int W_MMA = NPROD, W_SOFT = NPROD + 1, W_CONV = W_SOFT + NSOFT;
constexpr int NTHREADS = 32 * (W_CONV + NCONV);          // 512: four warps per scheduler, 128 registers
constexpr int GATHERS = TK / 4;                          // K gather groups (4 rows) per tile
constexpr uint32_t CODE_TILE = TK * 128;                 // 16 KB of E4M3 codes
constexpr uint32_t STAGE = 2 * CODE_TILE + 2 * TK * 4;   // K codes, V codes, K scales, V scales
constexpr uint32_t VH_TILE = TK * 128 * 2;               // 32 KB FP16 V: two 64-d column atoms of 16 KB
constexpr uint32_t P_ATOM = 64 * 128;                    // 64 rows x 64 keys FP16 (8 KB)
constexpr uint32_t P_TILE = 2 * P_ATOM;                  // 64 rows x 128 keys
constexpr uint32_t QP_BYTES = 16 * 128;                  // 16 rows x 128 d E4M3
constexpr uint32_t OFF_STAGE = 0;
constexpr uint32_t OFF_VH = OFF_STAGE + NS * STAGE;
constexpr uint32_t OFF_P = OFF_VH + VH_TILE;
constexpr uint32_t OFF_QP = OFF_P + 2 * P_TILE;
constexpr uint32_t OFF_SLOT = OFF_QP + QP_BYTES;
constexpr uint32_t OFF_XA = OFF_SLOT + 2 * SLOT_CAP * 4; // int [2][4 quarters][8 heads]: tile maxima
constexpr uint32_t OFF_SCL = OFF_XA + 2 * 4 * 8 * 4;     // float [2][8 blocks][8 heads]: block factors 2^E
constexpr uint32_t OFF_FLAG = OFF_SCL + 2 * 8 * 8 * 4;   // int [2][8] votes, int [8] final vote
constexpr uint32_t OFF_FQ = OFF_FLAG + 128;              // float [8]: query multipliers
constexpr uint32_t OFF_LRED = OFF_FQ + 32;               // float [4 quarters][8 heads]: row sums
constexpr uint32_t OFF_BAR = OFF_LRED + 128;
constexpr int NBAR = 3 * NS + 14;
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;        // TMEM base address, abort flag
constexpr uint32_t SMEM_USED = OFF_MISC + 16;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;        // slack to align the base to 1024 B
static_assert(STAGE % 1024 == 0 && OFF_VH % 1024 == 0 && OFF_P % 1024 == 0 && OFF_QP % 1024 == 0, "alignment");
static_assert(OFF_SCL % 16 == 0 && OFF_XA % 16 == 0 && OFF_LRED % 16 == 0 && OFF_BAR % 8 == 0, "alignment");
static_assert(SMEM_ALLOC <= 232448, "decode_tc shared memory");

constexpr int B_FULL = 0;              // [NS] K codes and scales: NPROD arrivals + the gathered K bytes
// Consumer groups arrive once per warp (lane 0, after __syncwarp): counts are in warps.
constexpr int B_EMPTY = NS;            // [NS] 4 converter + 8 softmax warps
constexpr int B_QREADY = 2 * NS;       //      8: query pieces written, P' cleared
constexpr int B_SFULL = 2 * NS + 1;    // [2]  1: QK committed
constexpr int B_SFREE = 2 * NS + 3;    // [2]  8: S read
constexpr int B_VHFULL = 2 * NS + 5;   //      4: FP16 V written
constexpr int B_VHFREE = 2 * NS + 6;   //      1: PV committed (FP16 V consumed)
constexpr int B_PFULL = 2 * NS + 7;    // [2]  8: P' written
constexpr int B_DFULL = 2 * NS + 9;    // [2]  1: PV committed
constexpr int B_DFREE = 2 * NS + 11;   // [2]  8: D folded
constexpr int B_DRAIN = 2 * NS + 13;   //      1: every MMA finished
constexpr int B_FULLV = 2 * NS + 14;   // [NS] V codes: NPROD arrivals + the gathered V bytes
static_assert(B_DRAIN < B_FULLV && B_FULLV + NS <= NBAR, "barrier count");
constexpr int FULL_COUNT = NPROD;       // one arrival per producer warp (after its scale stores)
constexpr int BAR_SOFT = 1, BAR_PROD = 2;  // named barriers (0 is __syncthreads)

constexpr uint32_t TMEM_COLS = 256;    // S0 [0,16) S1 [16,32) D0 [64,128) D1 [128,192)
constexpr uint32_t TM_S = 0, TM_D = 64;
constexpr unsigned long long WAIT_LIMIT_NS = 4000000000ull;

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
__device__ __forceinline__ void mbar_expect_tx_only(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// try_wait with a suspend-time hint: the warp sleeps in hardware until the phase completes (or the hint
// runs out), instead of spinning and taking issue slots from the warps that do the work.
constexpr uint32_t SUSPEND_HINT_NS = 100000;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(SUSPEND_HINT_NS)
      : "memory");
  return ok != 0;
}
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err,
                                            bool honor_abort) {
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (honor_abort && *abort_flag) return false;
    if (globaltimer() - t0 > WAIT_LIMIT_NS) {
      *abort_flag = 1;
      flag_error(err, kDevErrTimeout);
      return false;
    }
  }
}
// Bounded wait.  With honor_abort, gives up as soon as another role of the CTA has timed out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err,
                                          bool honor_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag, err, honor_abort);
}
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Named barrier that also returns the AND of v over the participating threads.
__device__ __forceinline__ bool named_bar_and(int id, int count, bool v) {
  int r;
  asm volatile("{ .reg .pred p, q; setp.ne.s32 p, %1, 0; bar.red.and.pred q, %2, %3, p; selp.s32 %0, 1, 0, q; }"
               : "=r"(r)
               : "r"(static_cast<int>(v)), "r"(id), "r"(count)
               : "memory");
  return r != 0;
}
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, uint32_t bar, int r0, int r1,
                                            int r2, int r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Shared-memory matrix descriptor, 128-byte swizzle (start, leading and stride byte offsets >> 4).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}
// Instruction descriptors (FP32 accumulate).  QK: E4M3 x E4M3, both K-major, M = 128, N = 16.
// PV: F16 x F16, A MN-major (V^T, d contiguous), B K-major (P'), M = 128, N = 64.
constexpr uint32_t IDESC_QK = (1u << 4) | (0u << 7) | (0u << 10) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t IDESC_PV =
    (1u << 4) | (0u << 7) | (0u << 10) | (1u << 15) | ((64u >> 3) << 17) | ((128u >> 4) << 24);

__device__ __forceinline__ void umma_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void umma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ int redux_max_s32(int v) {
  int r;
  asm volatile("redux.sync.max.s32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}
// Order-preserving map between FP32 and int32, so a float maximum can use the integer reduction.
__device__ __forceinline__ int f2ord(float f) {
  const int b = __float_as_int(f);
  return b >= 0 ? b : (b ^ 0x7FFFFFFF);
}
__device__ __forceinline__ float ord2f(int o) { return __int_as_float(o >= 0 ? o : (o ^ 0x7FFFFFFF)); }

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled tile of 128-byte rows.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4);
}

__global__ void __launch_bounds__(NTHREADS, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const DecodeArgs a) {
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + OFF_MISC + 4);
  auto bar = [&](int i) { return base + OFF_BAR + 8u * i; };
  auto stage_k = [&](int s) { return base + OFF_STAGE + s * STAGE; };
  auto stage_v = [&](int s) { return base + OFF_STAGE + s * STAGE + CODE_TILE; };
  auto stage_ks = [&](int s) { return base + OFF_STAGE + s * STAGE + 2 * CODE_TILE; };
  auto stage_vs = [&](int s) { return base + OFF_STAGE + s * STAGE + 2 * CODE_TILE + TK * 4; };

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- the first window of slot indices, requested before the request geometry is known: the table
  // row holds req_stride entries, so the copy stays in bounds whatever seq_lens says ----
  if (warp < NPROD) {
    const int64_t j0p = static_cast<int64_t>(split) * a.chunk;
    int64_t cnt = a.req_stride - j0p;
    cnt = cnt < a.chunk ? cnt : a.chunk;
    cnt = cnt < SLOT_CAP ? cnt : SLOT_CAP;
    const int32_t* src = a.req_to_slot + static_cast<int64_t>(b) * a.req_stride + j0p;
    for (int k = threadIdx.x; k < cnt; k += 32 * NPROD) cp_async_4(base + OFF_SLOT + 4 * k, src + k);
  }

  // ---- request geometry (the same checks and conventions as the warp-level kernel) ----
  int64_t n = a.seq_lens[b];
  {
    const int64_t nmax = a.max_seq_len < a.req_stride ? a.max_seq_len : a.req_stride;
    if (n < 0 || n > nmax) {
      if (threadIdx.x == 0 && split == 0 && h == 0) flag_error(a.err, kDevErrSeqLen);
      n = n < 0 ? 0 : nmax;
    }
  }
  int64_t row0;
  int R;
  if (a.q_row_offsets) {
    row0 = a.q_row_offsets[b];
    R = a.q_row_offsets[b + 1] - a.q_row_offsets[b];
  } else {
    row0 = b;
    R = 1;
  }
  if (R < 0 || R > 1 || row0 < 0 || row0 + R > a.total_q_rows) {
    if (threadIdx.x == 0 && split == 0 && h == 0) flag_error(a.err, kDevErrQRows);
    cp_async_wait_all();
    return;
  }
  if (R == 0) {
    cp_async_wait_all();
    return;
  }
  if (n == 0) {  // nothing to attend to: the output row is zero
    if (split == 0)
      for (int i = threadIdx.x; i < a.group * kHeadDim; i += blockDim.x)
        a.out[(row0 * a.num_q_heads + h * a.group + i / kHeadDim) * kHeadDim + i % kHeadDim] = 0;
    cp_async_wait_all();
    return;
  }
  const int64_t j0l = static_cast<int64_t>(split) * a.chunk;
  if (j0l >= n) {
    cp_async_wait_all();
    return;
  }
  const int j0 = static_cast<int>(j0l);
  const int j1 = (j0l + a.chunk < n) ? static_cast<int>(j0l + a.chunk) : static_cast<int>(n);
  const int nkeys = j1 - j0;
  const int nT = (nkeys + TK - 1) / TK;
  const int G = a.group;

  // ---- set-up: barriers, TMEM ----
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; s++) {
      mbar_init(bar(B_FULL + s), FULL_COUNT);
      mbar_init(bar(B_FULLV + s), FULL_COUNT);
      mbar_init(bar(B_EMPTY + s), NCONV + NSOFT);
    }
    mbar_init(bar(B_QREADY), NSOFT);
    mbar_init(bar(B_VHFULL), NCONV);
    mbar_init(bar(B_VHFREE), 1);
    for (int x = 0; x < 2; x++) {
      mbar_init(bar(B_SFULL + x), 1);
      mbar_init(bar(B_SFREE + x), NSOFT);
      mbar_init(bar(B_PFULL + x), NSOFT);
      mbar_init(bar(B_DFULL + x), 1);
      mbar_init(bar(B_DFREE + x), NSOFT);
    }
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == W_MMA) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(base + OFF_MISC),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + OFF_MISC);

  if (warp < NPROD) {
    // ======================= producers: TMA gathers of K and V, scales through registers =====================
    const int pt = threadIdx.x;  // 0 .. 32 NPROD - 1
    const uint32_t sslot = base + OFF_SLOT;
    const int32_t* sslot_p = reinterpret_cast<const int32_t*>(gbase + OFF_SLOT);
    const int32_t* req = a.req_to_slot + static_cast<int64_t>(b) * a.req_stride + j0;
    auto row_of = [&](int key) -> int {  // pool row of key (relative to the slice); bad slots read slot 0
      int32_t slot = sslot_p[key % (2 * SLOT_CAP)];
      if (slot < 0 || slot >= a.num_rows) {
        flag_error(a.err, kDevErrBadSlot);
        slot = 0;
      }
      return static_cast<int>(static_cast<int64_t>(slot) * a.num_kv_heads + h);
    };
    // the scales of keys r = pt, pt + 32 NPROD, ... of a tile, loaded one tile ahead into registers
    constexpr int SPT = (TK + 32 * NPROD - 1) / (32 * NPROD);
    float ksn[SPT], vsn[SPT];
    auto load_scales = [&](int i) {
#pragma unroll
      for (int u = 0; u < SPT; u++) {
        const int r = pt + u * 32 * NPROD;
        ksn[u] = 0.0f;
        vsn[u] = 0.0f;
        if (r < TK && i * TK + r < nkeys) {
          const int row = row_of(i * TK + r);
          ksn[u] = __ldg(a.k_scales + row);
          vsn[u] = __ldg(a.v_scales + row);
        }
      }
    };
    cp_async_wait_all();  // the first window of slot indices, requested at entry
    named_bar_sync(BAR_PROD, 32 * NPROD);
    load_scales(0);
    int issued = 0;
    for (int i = 0; i < nT; i++) {
      const int s = i % NS;
      const int key0 = i * TK;
      bool w = true;
      if (i >= NS) w = mbar_wait(bar(B_EMPTY + s), ((i / NS) - 1) & 1, abort_flag, a.err);
      if (!named_bar_and(BAR_PROD, 32 * NPROD, w)) break;  // also: every producer is done with the last tile
      // The next tile starts a new window of slot indices: stage it in the other half of the double window
      // (that half's last reads were a whole window ago, before the barriers above).
      if ((key0 + TK) % SLOT_CAP == 0 && key0 + TK < nkeys) {
        const int k1 = key0 + TK;
        const int wn = (nkeys - k1 < SLOT_CAP) ? nkeys - k1 : SLOT_CAP;
        for (int k = pt; k < wn; k += 32 * NPROD) cp_async_4(sslot + 4 * ((k1 + k) % (2 * SLOT_CAP)), req + k1 + k);
        cp_async_wait_all();
        named_bar_sync(BAR_PROD, 32 * NPROD);
      }
      // Gather groups g = warp + NPROD * lane (keys 4g .. 4g+3 of the tile), spread over the warps.  K first,
      // on its own barrier, so QK and the softmax can start while the V rows are still on their way; the
      // bytes are announced before the gathers, and the K barrier's arrival waits for the scale stores.
      const uint32_t gbytes = 512u * ((GATHERS - warp + NPROD - 1) / NPROD);
      const bool has_group = warp + NPROD * lane < GATHERS;
      const int g = warp + NPROD * lane;
      int rows[4];
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const int key = key0 + 4 * g + e;
        rows[e] = (has_group && key < nkeys) ? row_of(key) : h;  // padding key: (slot 0, head h)
      }
      if (lane == 0) mbar_expect_tx_only(bar(B_FULL + s), gbytes);
      __syncwarp();
      if (has_group) tma_gather4(stage_k(s) + g * 512, &tmk, bar(B_FULL + s), rows[0], rows[1], rows[2], rows[3]);
      if (lane == 0) mbar_expect_tx(bar(B_FULLV + s), gbytes);
      __syncwarp();
      if (has_group) tma_gather4(stage_v(s) + g * 512, &tmv, bar(B_FULLV + s), rows[0], rows[1], rows[2], rows[3]);
      // this tile's scales (loaded one iteration ago) into the stage, then the next tile's into registers
#pragma unroll
      for (int u = 0; u < SPT; u++) {
        const int r = pt + u * 32 * NPROD;
        if (r < TK) {
          st_shared_u32(stage_ks(s) + r * 4, __float_as_uint(ksn[u]));
          st_shared_u32(stage_vs(s) + r * 4, __float_as_uint(vsn[u]));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_FULL + s));
      if (i + 1 < nT) load_scales(i + 1);
      issued = i + 1;
    }
    // every load issued must land before the CTA may exit
    for (int i = (issued > NS ? issued - NS : 0); i < issued; i++) {
      mbar_wait(bar(B_FULL + i % NS), (i / NS) & 1, abort_flag, a.err, false);
      mbar_wait(bar(B_FULLV + i % NS), (i / NS) & 1, abort_flag, a.err, false);
    }
  } else if (warp == W_MMA) {
    if (lane == 0) {
      // ======================= MMA issuer =======================
      bool ok = mbar_wait(bar(B_QREADY), 0, abort_flag, a.err);
      const uint32_t qp = base + OFF_QP;
      auto issue_pv = [&](int i) -> bool {
        const int x = i & 1;
        if (!mbar_wait(bar(B_PFULL + x), (i >> 1) & 1, abort_flag, a.err)) return false;
        if (!mbar_wait(bar(B_VHFULL), i & 1, abort_flag, a.err)) return false;
        if (i >= 2 && !mbar_wait(bar(B_DFREE + x), ((i >> 1) - 1) & 1, abort_flag, a.err)) return false;
        tc_fence_after();
        const uint32_t vh = base + OFF_VH, pt = base + OFF_P + x * P_TILE;
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          // A = V^T, MN-major: a k-step is 16 key rows (2 KB); the two 64-d column atoms are 16 KB apart.
          const uint64_t ad = sw128_desc(vh + kk * 2048, VH_TILE / 2, 1024);
          // B = P', K-major: 64 rows of 64 keys per 8 KB atom; a k-step is 32 bytes within the atom.
          const uint64_t bd = sw128_desc(pt + (kk >> 2) * P_ATOM + (kk & 3) * 32, 16, 1024);
          umma_f16(tmem + TM_D + x * 64, ad, bd, IDESC_PV, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(B_VHFREE));
        umma_commit(bar(B_DFULL + x));
        return true;
      };
      for (int i = 0; ok && i < nT; i++) {
        const int s = i % NS, x = i & 1;
        if (!mbar_wait(bar(B_FULL + s), (i / NS) & 1, abort_flag, a.err)) {
          ok = false;
          break;
        }
        if (i >= 2 && !mbar_wait(bar(B_SFREE + x), ((i >> 1) - 1) & 1, abort_flag, a.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; kk++)
          umma_f8(tmem + TM_S + x * 16, sw128_desc(stage_k(s) + kk * 32, 16, 1024), sw128_desc(qp + kk * 32, 16, 1024),
                  IDESC_QK, kk > 0 ? 1u : 0u);
        umma_commit(bar(B_SFULL + x));
        if (i >= 1 && !issue_pv(i - 1)) {
          ok = false;
          break;
        }
      }
      if (ok) issue_pv(nT - 1);
      umma_commit(bar(B_DRAIN));
      mbar_wait(bar(B_DRAIN), 0, abort_flag, a.err, false);
    }
  } else if (warp >= W_CONV) {
    // ======================= V converter: E4M3 codes -> FP16, MN-major SW128 =======================
    const int ct = threadIdx.x - 32 * W_CONV;  // key rows ct, ct + 32 NCONV, ...
    for (int i = 0; i < nT; i++) {
      const int s = i % NS;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_FULLV + s), (i / NS) & 1, abort_flag, a.err))) break;
      if (i >= 1 && !__all_sync(0xffffffffu, mbar_wait(bar(B_VHFREE), (i - 1) & 1, abort_flag, a.err))) break;
      const uint32_t src = stage_v(s), dst = base + OFF_VH;
      for (int t = ct; t < TK; t += 32 * NCONV) {
      const uint32_t keep = (i * TK + t < nkeys) ? 0xFFFFFFFFu : 0u;  // padding keys: V row of zeros
#pragma unroll
      for (int c = 0; c < 8; c++) {
        const uint4 w = ld_shared_v4(src + sw128(t, c));  // codes of d = 16c .. 16c+15
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
        uint32_t hv[8];
#pragma unroll
        for (int q = 0; q < 4; q++) {
          hv[2 * q] = e4m3_lo2(ww[q]) & keep;
          hv[2 * q + 1] = e4m3_hi2(ww[q]) & keep;
        }
#pragma unroll
        for (int hh = 0; hh < 2; hh++) {  // FP16 chunk 2c + hh holds d = 16c + 8hh .. +7
          const int ch = 2 * c + hh;
          const uint32_t addr = dst + (ch >> 3) * (VH_TILE / 2) + sw128(t, ch & 7);
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(hv[4 * hh]), "r"(hv[4 * hh + 1]),
                       "r"(hv[4 * hh + 2]), "r"(hv[4 * hh + 3])
                       : "memory");
        }
      }
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(B_VHFULL));
        mbar_arrive(bar(B_EMPTY + s));
      }
    }
  } else {
    // ======================= softmax warps =======================
    // A warp reaches TMEM lanes 32 (warp % 4) .. +31 only: thread t is key row t of S and d row t of D.
    // Warps W_SOFT .. +3 take heads 0-3, the next four heads 4-7.
    const int qd = warp & 3;
    const int wi = warp - W_SOFT;        // 0..7
    const int hh = wi >> 2;              // head half
    const int t = qd * 32 + lane;
    const int st = threadIdx.x - 32 * W_SOFT;  // 0..255
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(qd * 32) << 16);
    int* xa = reinterpret_cast<int*>(gbase + OFF_XA);
    float* scl = reinterpret_cast<float*>(gbase + OFF_SCL);
    volatile int* vote = reinterpret_cast<volatile int*>(gbase + OFF_FLAG);
    float* fqs = reinterpret_cast<float*>(gbase + OFF_FQ);
    float* lred = reinterpret_cast<float*>(gbase + OFF_LRED);

    // --- query pieces (threads st < 128: head g = st / 16, d = 8 (st % 16) .. +7); P' cleared ---
    if (st < 128) {
      const int g = st >> 4, d0 = (st & 15) * 8;
      float qv[8];
      float amax = 0.0f;
      if (g < G) {
        const uint4 v =
            __ldg(reinterpret_cast<const uint4*>(a.q + (row0 * a.num_q_heads + h * G + g) * kHeadDim + d0));
        const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; e++) {
          qv[2 * e] = bf16_lo(vv[e]);
          qv[2 * e + 1] = bf16_hi(vv[e]);
        }
#pragma unroll
        for (int e = 0; e < 8; e++) amax = fmaxf(amax, fabsf(qv[e]));
      } else {
#pragma unroll
        for (int e = 0; e < 8; e++) qv[e] = 0.0f;
      }
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      int ex = (amax > 0.0f) ? ilogbf(amax) : 0;
      ex = ex < -120 ? -120 : ex;
      // x = q 2^(7-ex) has |x| < 256; pieces x = h1 + h2/16 (exact unless |q| < 2^-13 max|q|)
      const float up = __uint_as_float(static_cast<uint32_t>(127 + 7 - ex) << 23);
      uint32_t hi[2], lo[2];
#pragma unroll
      for (int e = 0; e < 8; e += 4) {
        const float x0 = qv[e] * up, x1 = qv[e + 1] * up, x2 = qv[e + 2] * up, x3 = qv[e + 3] * up;
        const uint32_t c01 = e4m3x2_encode(x0, x1), c23 = e4m3x2_encode(x2, x3);
        const float2 v01 = f16x2_to_float2(e4m3x2_to_f16x2(c01)), v23 = f16x2_to_float2(e4m3x2_to_f16x2(c23));
        hi[e >> 2] = c01 | (c23 << 16);
        lo[e >> 2] = e4m3x2_encode((x0 - v01.x) * 16.0f, (x1 - v01.y) * 16.0f) |
                     (e4m3x2_encode((x2 - v23.x) * 16.0f, (x3 - v23.y) * 16.0f) << 16);
      }
      // rows g (first piece) and 8 + g (second piece) of the K-major SW128 operand, bytes d0 .. d0+7
      const uint32_t qp = base + OFF_QP;
      asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(qp + sw128(g, d0 >> 4) + (d0 & 15)), "r"(hi[0]),
                   "r"(hi[1])
                   : "memory");
      asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(qp + sw128(8 + g, d0 >> 4) + (d0 & 15)), "r"(lo[0]),
                   "r"(lo[1])
                   : "memory");
      if ((st & 15) == 0)
        fqs[g] = (g < G) ? __uint_as_float(static_cast<uint32_t>(127 - 7 + ex) << 23) * a.qk_scale_log2 : 0.0f;
    }
    // P' is zero outside each key's own (half, block, head) rows: clear both buffers once
    for (int k = st; k < static_cast<int>(2 * P_TILE / 16); k += 32 * NSOFT) st_shared_zero16(base + OFF_P + 16 * k);
    fence_proxy_async();
    named_bar_sync(BAR_SOFT, 32 * NSOFT);
    if (lane == 0) mbar_arrive(bar(B_QREADY));

    float fq[4], m[4], lsum[4], O[4], alpha_prev[4];
#pragma unroll
    for (int gg = 0; gg < 4; gg++) {
      fq[gg] = fqs[hh * 4 + gg];
      m[gg] = -INFINITY;
      lsum[gg] = 0.0f;
      O[gg] = 0.0f;
      alpha_prev[gg] = 1.0f;
    }

    // O = O alpha_i + sum over the 8 blocks of D_i[half, block, head] 2^(E[block, head] - 127)
    auto fold = [&](int i) -> bool {
      const int x = i & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_DFULL + x), (i >> 1) & 1, abort_flag, a.err))) return false;
      tc_fence_after();
      uint32_t dv[32];
      tmem_ld32(lane_base + TM_D + x * 64 + hh * 32, dv);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DFREE + x));
      const float4* sc4 = reinterpret_cast<const float4*>(scl + x * 64 + hh * 4);
      float acc[4];
#pragma unroll
      for (int gg = 0; gg < 4; gg++) acc[gg] = O[gg] * alpha_prev[gg];
#pragma unroll
      for (int blk = 0; blk < 8; blk++) {
        const float4 f = sc4[blk * 2];  // scl[x][blk][hh*4 .. hh*4+3]
        acc[0] = fmaf(__uint_as_float(dv[blk * 4 + 0]), f.x, acc[0]);
        acc[1] = fmaf(__uint_as_float(dv[blk * 4 + 1]), f.y, acc[1]);
        acc[2] = fmaf(__uint_as_float(dv[blk * 4 + 2]), f.z, acc[2]);
        acc[3] = fmaf(__uint_as_float(dv[blk * 4 + 3]), f.w, acc[3]);
      }
#pragma unroll
      for (int gg = 0; gg < 4; gg++) O[gg] = acc[gg];
      return true;
    };

    bool ok = true;
    int done = 0;  // tiles whose P' has been handed to the MMA warp
    for (int i = 0; i < nT; i++) {
      const int s = i % NS, x = i & 1;
      bool w = ok && mbar_wait(bar(B_FULL + s), (i / NS) & 1, abort_flag, a.err);
      w = w && mbar_wait(bar(B_SFULL + x), (i >> 1) & 1, abort_flag, a.err);
      w = __all_sync(0xffffffffu, w);
      const bool valid = i * TK + t < nkeys;
      float sg[4], sv = 0.0f;
      if (w) {
        tc_fence_after();
        uint32_t sc[16];
        tmem_ld16(lane_base + TM_S + x * 16, sc);
        const float sk = ld_shared_f32(stage_ks(s) + t * 4);
        sv = ld_shared_f32(stage_vs(s) + t * 4);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(B_SFREE + x));
          mbar_arrive(bar(B_EMPTY + s));
        }
#pragma unroll
        for (int gg = 0; gg < 4; gg++) {
          const int g = hh * 4 + gg;
          sg[gg] = valid ? fmaf(__uint_as_float(sc[8 + g]), 1.0f / 16.0f, __uint_as_float(sc[g])) * (sk * fq[gg])
                         : -INFINITY;
        }
      } else {
#pragma unroll
        for (int gg = 0; gg < 4; gg++) sg[gg] = -INFINITY;
      }
      // exact tile maximum of s per head over the 128 keys; the vote rides on the same barrier
      int om[4];
#pragma unroll
      for (int gg = 0; gg < 4; gg++) om[gg] = redux_max_s32(f2ord(sg[gg]));
      if (lane == 0) {
        *reinterpret_cast<int4*>(xa + x * 32 + qd * 8 + hh * 4) = make_int4(om[0], om[1], om[2], om[3]);
        vote[x * 8 + wi] = w ? 1 : 0;
      }
      named_bar_sync(BAR_SOFT, 32 * NSOFT);
      bool all = true;
#pragma unroll
      for (int k = 0; k < NSOFT; k++) all = all && vote[x * 8 + k];
      if (!all) {
        ok = false;
        break;
      }
      float alpha[4], wv[4];
      uint32_t pk = 0;  // biased exponents of w, one byte per head
#pragma unroll
      for (int gg = 0; gg < 4; gg++) {
        const int* xg = xa + x * 32 + hh * 4 + gg;
        const float mt = ord2f(max(max(xg[0], xg[8]), max(xg[16], xg[24])));
        const float mn = fmaxf(m[gg], mt);
        const float mu = (mn == -INFINITY) ? 0.0f : mn;
        alpha[gg] = fast_exp2(m[gg] - mu);
        m[gg] = mn;
        const float p = valid ? fast_exp2(sg[gg] - mu) : 0.0f;
        lsum[gg] = fmaf(lsum[gg], alpha[gg], p);
        wv[gg] = valid ? p * sv : 0.0f;
        pk |= (__float_as_uint(wv[gg]) >> 23) << (8 * gg);
      }
      // block maxima over the 16 keys of this half-warp (bytewise unsigned max), clamped to [1, 253]
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) pk = __vmaxu4(pk, __shfl_xor_sync(0xffffffffu, pk, off));
      pk = __vminu4(__vmaxu4(pk, 0x01010101u), 0xFDFDFDFDu);
      const int blk = t >> 4;
      if ((lane & 15) == 0) {
        float4 f;
        f.x = __uint_as_float((pk & 0xFFu) << 23);
        f.y = __uint_as_float(((pk >> 8) & 0xFFu) << 23);
        f.z = __uint_as_float(((pk >> 16) & 0xFFu) << 23);
        f.w = __uint_as_float((pk >> 24) << 23);
        *reinterpret_cast<float4*>(scl + x * 64 + blk * 8 + hh * 4) = f;
      }
      // P'[(hh, blk, gg)][t] = w 2^(127 - E) in FP16 (K-major SW128: 64-key atoms, row 32 hh + 4 blk + gg)
      const uint32_t pt = base + OFF_P + x * P_TILE + (t >> 6) * P_ATOM;
      const int kc = t & 63;
#pragma unroll
      for (int gg = 0; gg < 4; gg++) {
        const uint32_t e = (pk >> (8 * gg)) & 0xFFu;
        const __half hv = __float2half_rn(wv[gg] * __uint_as_float((254u - e) << 23));
        const uint32_t addr = pt + sw128(hh * 32 + blk * 4 + gg, kc >> 3) + (kc & 7) * 2;
        asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(__half_as_ushort(hv)) : "memory");
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL + x));
      done = i + 1;
      // fold the previous tile (its block factors were published before this tile's barrier)
      if (i >= 1) ok = fold(i - 1);
#pragma unroll
      for (int gg = 0; gg < 4; gg++) alpha_prev[gg] = alpha[gg];
    }
    // final vote: the last tile's block factors become visible at this barrier too
    if (lane == 0) vote[16 + wi] = (ok && done == nT) ? 1 : 0;
    named_bar_sync(BAR_SOFT, 32 * NSOFT);
    bool all_ok = true;
#pragma unroll
    for (int k = 0; k < NSOFT; k++) all_ok = all_ok && vote[16 + k];
    if (all_ok) fold(nT - 1);

    // ---- partial (m, l, O) of this slice per query head; thread t = d ----
#pragma unroll
    for (int gg = 0; gg < 4; gg++)
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) lsum[gg] += __shfl_xor_sync(0xffffffffu, lsum[gg], off);
    if (lane == 0)
      *reinterpret_cast<float4*>(lred + qd * 8 + hh * 4) = make_float4(lsum[0], lsum[1], lsum[2], lsum[3]);
    named_bar_sync(BAR_SOFT, 32 * NSOFT);
#pragma unroll
    for (int gg = 0; gg < 4; gg++) {
      const int g = hh * 4 + gg;
      if (g < G) {
        const int64_t prow = ((row0 * a.num_q_heads) + h * G + g) * a.num_splits + split;
        a.part_acc[prow * kHeadDim + t] = O[gg];
        if (t == 0) {
          a.part_ml[prow * 2] = m[gg];
          a.part_ml[prow * 2 + 1] = lred[g] + lred[8 + g] + lred[16 + g] + lred[24 + g];
        }
      }
    }
  }

  // ======================= teardown, then the merge by the last slice to arrive =======================
  tc_fence_before();
  __syncthreads();
  if (warp == W_MMA) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
  __shared__ int s_last;
  const int64_t nsl64 = (n + a.chunk - 1) / a.chunk;
  const int nslices = static_cast<int>(nsl64 < a.num_splits ? nsl64 : a.num_splits);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int* ctr = a.counters + static_cast<int64_t>(b) * a.num_kv_heads + h;
    const int prev = atomicAdd(ctr, 1);
    s_last = (prev == nslices - 1);
    if (s_last) *ctr = 0;  // ready for the next call
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  merge_split_partials(a, row0, 1, h, nslices, gbase, OFF_SLOT);  // everything below the slots is idle now
}

// ---------------------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// One pool code tensor as a 2-D byte tensor: rows = (slot, KV head) of 128 bytes.  Gather boxes are one
// row high and 128 bytes wide, 128-byte swizzle.
bool make_row_map(CUtensorMap* m, const void* ptr, int64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, 1};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t s) {
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int64_t rows = a.num_rows * a.num_kv_heads;  // gather row coordinates are int32
  if (rows >= (int64_t(1) << 31) - 1) return cudaErrorInvalidValue;
  CUtensorMap tmk, tmv;
  if (!make_row_map(&tmk, a.k_codes, rows) || !make_row_map(&tmv, a.v_codes, rows)) return cudaErrorInvalidValue;
  dim3 grid(a.num_splits, a.num_kv_heads, a.batch);
  return launch_k(decode_tc_kernel, grid, dim3(NTHREADS), SMEM_ALLOC, s, tmk, tmv, a);
}

}  // namespace ftkv
