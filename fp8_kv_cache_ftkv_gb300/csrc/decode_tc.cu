// decode_tc.cu -- single-row split-K decode attention on the tcgen05 tensor cores, fed by TMA gathers.
//
// What it computes (FreeToken PR #897, opening description and "Fresh R9700 stage-1 A/B"): for each
// query head i (KV head h = i / G) of a request with n cached keys,
//     o = sum_j softmax_j((q . k^_j) * sm_scale) v^_j,   k^_j = decode(codeK_j) scaleK_j, v^_j likewise,
// split over key slices whose partials (m, l, O) are merged by the slice that finishes last (the same
// partial format and merge as the warp-level kernel in decode.cu).  This kernel serves requests with
// one query row; the warp-level kernel serves the multi-row (MTP / speculative) case.
//
// CTA = (key slice, KV head, request), 320 threads, tiles of 128 keys:
//   warp 0      TMEM allocation; producer: stages the slice's slot indices in shared memory, then per
//               tile each lane issues one TMA tile::gather4 for 4 K code rows and one for the same 4 V
//               code rows (128 B each, 128-byte swizzle) plus cp.async copies of their 8 scales, all
//               completing on one mbarrier (3-stage ring).  Padding keys past the slice's end gather
//               the head's row of slot 0 (always in bounds); they get no scales, the softmax gives them
//               weight 0 by selection and the converter writes their V rows as zeros.
//   warp 1      lane 0 issues the MMAs:
//                 S_i = K_i Qp^T    kind::f8f6f4, E4M3 x E4M3 -> FP32, M = 128 keys, N = 16 (8 query
//                                   heads x 2 exact E4M3 pieces of the BF16 query), K = 128 d; the
//                                   stored K codes are the A operand exactly as TMA left them.
//                 D_i = Vh_i^T P'_i kind::f16, M = 128 d, N = 64 (8 heads x 8 blocks of 16 keys),
//                                   K = 128 keys; V is the MN-major A operand.
//               S and D are double-buffered in TMEM.
//   warps 2..5  softmax, one thread per key row of S (= TMEM lane): scores, exact per-tile maxima per head
//               (redux.sync + one shared-memory exchange), p = 2^(s - m), the value-weighted weight
//               w = p scaleV, and P' = w 2^-E written in FP16 to row (block, head) of P', where 2^E is
//               the power of two of the block's largest w (each 16-key block keeps FP16's full range).
//               Then the fold O = O alpha_i + sum_blocks D_i[block] 2^E[block] in FP32 registers, one
//               thread per d row of D.
//   warps 6..9  convert the V code tile to FP16 (packed hardware converter) in the MN-major SW128 layout.
// Every mbarrier wait is bounded by %globaltimer; on expiry the CTA flags FTKV_DEVERR_TIMEOUT, drains its
// loads and MMAs, releases TMEM and leaves its outputs unspecified.  Named barriers among the softmax
// warps are only crossed with a CTA-uniform decision (a flag vote at each barrier), so a timeout cannot
// leave one warp waiting at a barrier the others skipped.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "ftkv_device.cuh"
#include "ftkv_internal.h"

namespace ftkv {
namespace {

constexpr int TK = 128;                                  // keys per tile
constexpr int NS = 3;                                    // stages of the gather ring
constexpr int SLOT_CAP = 2048;                           // slot indices staged per window
constexpr uint32_t CODE_TILE = TK * 128;                 // 16 KB of E4M3 codes
constexpr uint32_t STAGE = 2 * CODE_TILE + 2 * TK * 4;   // K codes, V codes, K scales, V scales
constexpr uint32_t VH_TILE = TK * 128 * 2;               // 32 KB FP16 V: two 64-d column atoms of 16 KB
constexpr uint32_t P_ATOM = 64 * 128;                    // 64 rows x 64 keys FP16 (8 KB)
constexpr uint32_t P_TILE = 2 * P_ATOM;                  // 64 rows (block, head) x 128 keys
constexpr uint32_t QP_BYTES = 16 * 128;                  // 16 rows x 128 d E4M3
constexpr uint32_t OFF_STAGE = 0;
constexpr uint32_t OFF_VH = OFF_STAGE + NS * STAGE;
constexpr uint32_t OFF_P = OFF_VH + 2 * VH_TILE;
constexpr uint32_t OFF_QP = OFF_P + 2 * P_TILE;
constexpr uint32_t OFF_SLOT = OFF_QP + QP_BYTES;
constexpr uint32_t OFF_XA = OFF_SLOT + SLOT_CAP * 4;     // int [2][4 warps][8 heads]: tile maxima
constexpr uint32_t OFF_EB = OFF_XA + 2 * 4 * 8 * 4;      // u32 [2][8 blocks][2]: block exponents, 1 byte/head
constexpr uint32_t OFF_FLAG = OFF_EB + 2 * 8 * 2 * 4;    // int [2][4] votes, int [4] final vote
constexpr uint32_t OFF_FQ = OFF_FLAG + 64;               // float [8]: query multipliers
constexpr uint32_t OFF_LRED = OFF_FQ + 32;               // float [4][8]: row sums
constexpr uint32_t OFF_BAR = OFF_LRED + 128;
constexpr int NBAR = 2 * NS + 16;
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;        // TMEM base address, abort flag
constexpr uint32_t SMEM_USED = OFF_MISC + 16;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;        // slack to align the base to 1024 B
static_assert(STAGE % 1024 == 0 && OFF_VH % 1024 == 0 && OFF_P % 1024 == 0 && OFF_QP % 1024 == 0, "alignment");
static_assert(SMEM_ALLOC <= 232448, "decode_tc shared memory");

constexpr int B_FULL = 0;              // [NS] 33: expect_tx + one cp.async arrival per producer lane
constexpr int B_EMPTY = NS;            // [NS] 256: converter + softmax threads
constexpr int B_QREADY = 2 * NS;       //      128: query pieces written
constexpr int B_SFULL = 2 * NS + 1;    // [2]  1: QK committed
constexpr int B_SFREE = 2 * NS + 3;    // [2]  128: S read
constexpr int B_VHFULL = 2 * NS + 5;   // [2]  128: FP16 V written
constexpr int B_VHFREE = 2 * NS + 7;   // [2]  1: PV committed (V and P' consumed)
constexpr int B_PFULL = 2 * NS + 9;    // [2]  128: P' written
constexpr int B_DFULL = 2 * NS + 11;   // [2]  1: PV committed
constexpr int B_DFREE = 2 * NS + 13;   // [2]  128: D folded
constexpr int B_DRAIN = 2 * NS + 15;   //      1: every MMA finished

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
// Bounded wait.  With honor_abort, gives up as soon as another role of the CTA has timed out.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err,
                                       bool honor_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
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
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
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
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,"
      "%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]),
        "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]),
        "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]),
        "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]),
        "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
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

__global__ void __launch_bounds__(320, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const DecodeArgs a) {
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
    return;
  }
  if (R == 0) return;
  if (n == 0) {  // nothing to attend to: the output row is zero
    if (split == 0)
      for (int i = threadIdx.x; i < a.group * kHeadDim; i += blockDim.x)
        a.out[(row0 * a.num_q_heads + h * a.group + i / kHeadDim) * kHeadDim + i % kHeadDim] = 0;
    return;
  }
  const int64_t j0l = static_cast<int64_t>(split) * a.chunk;
  if (j0l >= n) return;
  const int j0 = static_cast<int>(j0l);
  const int j1 = (j0l + a.chunk < n) ? static_cast<int>(j0l + a.chunk) : static_cast<int>(n);
  const int nkeys = j1 - j0;
  const int nT = (nkeys + TK - 1) / TK;
  const int G = a.group;

  // ---- set-up: barriers, TMEM ----
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; s++) {
      mbar_init(bar(B_FULL + s), 33);
      mbar_init(bar(B_EMPTY + s), 256);
    }
    mbar_init(bar(B_QREADY), 128);
    for (int x = 0; x < 2; x++) {
      mbar_init(bar(B_SFULL + x), 1);
      mbar_init(bar(B_SFREE + x), 128);
      mbar_init(bar(B_VHFULL + x), 128);
      mbar_init(bar(B_VHFREE + x), 1);
      mbar_init(bar(B_PFULL + x), 128);
      mbar_init(bar(B_DFULL + x), 1);
      mbar_init(bar(B_DFREE + x), 128);
    }
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(base + OFF_MISC),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + OFF_MISC);

  if (warp == 0) {
    // ======================= producer =======================
    const uint32_t sslot = base + OFF_SLOT;
    const int32_t* req = a.req_to_slot + static_cast<int64_t>(b) * a.req_stride + j0;
    const int32_t* sslot_p = reinterpret_cast<const int32_t*>(gbase + OFF_SLOT);
    int issued = 0;
    for (int i = 0; i < nT; i++) {
      const int s = i % NS;
      const int key0 = i * TK;
      if (key0 % SLOT_CAP == 0) {  // stage the next window of slot indices (the previous one is consumed)
        const int wn = (nkeys - key0 < SLOT_CAP) ? nkeys - key0 : SLOT_CAP;
        for (int k = lane; k < wn; k += 32) cp_async_4(sslot + 4 * k, req + key0 + k);
        cp_async_wait_all();
        __syncwarp();
      }
      if (i >= NS && !__all_sync(0xffffffffu, mbar_wait(bar(B_EMPTY + s), ((i / NS) - 1) & 1, abort_flag, a.err)))
        break;
      int rows[4];
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const int key = key0 + 4 * lane + e;
        int r = h;  // padding key: (slot 0, head h)
        if (key < nkeys) {
          int32_t slot = sslot_p[key % SLOT_CAP];
          if (slot < 0 || slot >= a.num_rows) {  // flagged; row 0 keeps the read in bounds
            flag_error(a.err, kDevErrBadSlot);
            slot = 0;
          }
          r = static_cast<int>(static_cast<int64_t>(slot) * a.num_kv_heads + h);
        }
        rows[e] = r;
      }
      if (lane == 0) mbar_expect_tx(bar(B_FULL + s), 2 * CODE_TILE);
      __syncwarp();
      tma_gather4(stage_k(s) + lane * 512, &tmk, bar(B_FULL + s), rows[0], rows[1], rows[2], rows[3]);
      tma_gather4(stage_v(s) + lane * 512, &tmv, bar(B_FULL + s), rows[0], rows[1], rows[2], rows[3]);
#pragma unroll
      for (int e = 0; e < 4; e++) {
        if (key0 + 4 * lane + e < nkeys) {
          cp_async_4(stage_ks(s) + (4 * lane + e) * 4, a.k_scales + rows[e]);
          cp_async_4(stage_vs(s) + (4 * lane + e) * 4, a.v_scales + rows[e]);
        }
      }
      cp_async_arrive_noinc(bar(B_FULL + s));
      issued = i + 1;
    }
    // every load issued must land before the CTA may exit
    for (int i = (issued > NS ? issued - NS : 0); i < issued; i++)
      mbar_wait(bar(B_FULL + i % NS), (i / NS) & 1, abort_flag, a.err, false);
    cp_async_wait_all();
  } else if (warp == 1) {
    if (lane == 0) {
      // ======================= MMA issuer =======================
      bool ok = mbar_wait(bar(B_QREADY), 0, abort_flag, a.err);
      const uint32_t qp = base + OFF_QP;
      auto issue_pv = [&](int i) -> bool {
        const int x = i & 1;
        if (!mbar_wait(bar(B_PFULL + x), (i >> 1) & 1, abort_flag, a.err)) return false;
        if (!mbar_wait(bar(B_VHFULL + x), (i >> 1) & 1, abort_flag, a.err)) return false;
        if (i >= 2 && !mbar_wait(bar(B_DFREE + x), ((i >> 1) - 1) & 1, abort_flag, a.err)) return false;
        tc_fence_after();
        const uint32_t vh = base + OFF_VH + x * VH_TILE, pt = base + OFF_P + x * P_TILE;
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          // A = V^T, MN-major: a k-step is 16 key rows (2 KB); the two 64-d column atoms are 16 KB apart.
          const uint64_t ad = sw128_desc(vh + kk * 2048, VH_TILE / 2, 1024);
          // B = P', K-major: 64 rows of 64 keys per 8 KB atom; a k-step is 32 bytes within the atom.
          const uint64_t bd = sw128_desc(pt + (kk >> 2) * P_ATOM + (kk & 3) * 32, 16, 1024);
          umma_f16(tmem + TM_D + x * 64, ad, bd, IDESC_PV, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(B_VHFREE + x));
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
  } else if (warp >= 6) {
    // ======================= V converter: E4M3 codes -> FP16, MN-major SW128 =======================
    const int t = threadIdx.x - 192;  // key row
    for (int i = 0; i < nT; i++) {
      const int s = i % NS, x = i & 1;
      if (!mbar_wait(bar(B_FULL + s), (i / NS) & 1, abort_flag, a.err)) break;
      if (i >= 2 && !mbar_wait(bar(B_VHFREE + x), ((i >> 1) - 1) & 1, abort_flag, a.err)) break;
      const uint32_t src = stage_v(s), dst = base + OFF_VH + x * VH_TILE;
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
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(bar(B_VHFULL + x));
      mbar_arrive(bar(B_EMPTY + s));
    }
  } else {
    // ======================= softmax warps 2..5 =======================
    // A warp reaches TMEM lanes 32 (warp % 4) .. +31 only: thread t is key row t of S and d row t of D.
    const int wq = warp & 3;
    const int t = wq * 32 + lane;
    const int wi = warp - 2;  // slot in the exchange arrays
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    int* xa = reinterpret_cast<int*>(gbase + OFF_XA);
    uint32_t* ebw = reinterpret_cast<uint32_t*>(gbase + OFF_EB);
    volatile int* vote = reinterpret_cast<volatile int*>(gbase + OFF_FLAG);
    float* fqs = reinterpret_cast<float*>(gbase + OFF_FQ);
    float* lred = reinterpret_cast<float*>(gbase + OFF_LRED);

    // --- query pieces: thread -> head g = t / 16, d = 8 (t % 16) .. +7 ---
    {
      const int g = t >> 4, d0 = (t & 15) * 8;
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
      if ((t & 15) == 0)
        fqs[g] = (g < G) ? __uint_as_float(static_cast<uint32_t>(127 - 7 + ex) << 23) * a.qk_scale_log2 : 0.0f;
      // P' is zero outside each key's own (block, head) rows: clear both buffers once
      for (int k = t; k < static_cast<int>(2 * P_TILE / 16); k += 128) st_shared_zero16(base + OFF_P + 16 * k);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      named_bar_sync(1, 128);
      mbar_arrive(bar(B_QREADY));
    }
    float fq[8];
#pragma unroll
    for (int g = 0; g < 8; g++) fq[g] = fqs[g];

    float m[8], lsum[8], O[8], alpha_prev[8];
#pragma unroll
    for (int g = 0; g < 8; g++) {
      m[g] = -INFINITY;
      lsum[g] = 0.0f;
      O[g] = 0.0f;
      alpha_prev[g] = 1.0f;
    }

    // O = O alpha_i + sum over 16-key blocks of D_i[block] 2^(E[block] - 127)
    auto fold = [&](int i) -> bool {
      const int x = i & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_DFULL + x), (i >> 1) & 1, abort_flag, a.err))) return false;
      tc_fence_after();
      uint32_t dv[64];
      tmem_ld64(lane_base + TM_D + x * 64, dv);
      tc_fence_before();
      mbar_arrive(bar(B_DFREE + x));
      const uint32_t* eb = ebw + x * 16;
      float acc[8];
#pragma unroll
      for (int g = 0; g < 8; g++) acc[g] = O[g] * alpha_prev[g];
#pragma unroll
      for (int blk = 0; blk < 8; blk++) {
        const uint32_t e0 = eb[2 * blk], e1 = eb[2 * blk + 1];
#pragma unroll
        for (int g = 0; g < 8; g++) {
          const uint32_t e = ((g < 4 ? e0 : e1) >> (8 * (g & 3))) & 0xFFu;
          acc[g] = fmaf(__uint_as_float(dv[blk * 8 + g]), __uint_as_float(e << 23), acc[g]);
        }
      }
#pragma unroll
      for (int g = 0; g < 8; g++) O[g] = acc[g];
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
      float sg[8], sv = 0.0f;
      if (w) {
        tc_fence_after();
        uint32_t sc[16];
        tmem_ld16(lane_base + TM_S + x * 16, sc);
        tc_fence_before();
        mbar_arrive(bar(B_SFREE + x));
        const float sk = ld_shared_f32(stage_ks(s) + t * 4);
        sv = ld_shared_f32(stage_vs(s) + t * 4);
        mbar_arrive(bar(B_EMPTY + s));
#pragma unroll
        for (int g = 0; g < 8; g++)
          sg[g] = valid ? fmaf(__uint_as_float(sc[8 + g]), 1.0f / 16.0f, __uint_as_float(sc[g])) * (sk * fq[g])
                        : -INFINITY;
      } else {
#pragma unroll
        for (int g = 0; g < 8; g++) sg[g] = -INFINITY;
      }
      // exact tile maximum of s per head over the 128 keys; the vote rides on the same barrier
      int om[8];
#pragma unroll
      for (int g = 0; g < 8; g++) om[g] = redux_max_s32(f2ord(sg[g]));
      if (lane == 0) {
#pragma unroll
        for (int g = 0; g < 8; g++) xa[x * 32 + wi * 8 + g] = om[g];
        vote[x * 4 + wi] = w ? 1 : 0;
      }
      named_bar_sync(1, 128);
      if (!(vote[x * 4 + 0] && vote[x * 4 + 1] && vote[x * 4 + 2] && vote[x * 4 + 3])) {
        ok = false;
        break;
      }
      float alpha[8], wv[8];
      uint32_t pk0 = 0, pk1 = 0;  // biased exponents of w, one byte per head
#pragma unroll
      for (int g = 0; g < 8; g++) {
        const int* xg = xa + x * 32 + g;
        const float mt = ord2f(max(max(xg[0], xg[8]), max(xg[16], xg[24])));
        const float mn = fmaxf(m[g], mt);
        const float mu = (mn == -INFINITY) ? 0.0f : mn;
        alpha[g] = fast_exp2(m[g] - mu);
        m[g] = mn;
        const float p = valid ? fast_exp2(sg[g] - mu) : 0.0f;
        lsum[g] = fmaf(lsum[g], alpha[g], p);
        wv[g] = valid ? p * sv : 0.0f;
        const uint32_t eb = __float_as_uint(wv[g]) >> 23;
        if (g < 4) pk0 |= eb << (8 * g);
        else pk1 |= eb << (8 * (g - 4));
      }
      // block maxima over the 16 keys of this half-warp (bytewise unsigned max), clamped to [1, 253]
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) {
        pk0 = __vmaxu4(pk0, __shfl_xor_sync(0xffffffffu, pk0, off));
        pk1 = __vmaxu4(pk1, __shfl_xor_sync(0xffffffffu, pk1, off));
      }
      pk0 = __vminu4(__vmaxu4(pk0, 0x01010101u), 0xFDFDFDFDu);
      pk1 = __vminu4(__vmaxu4(pk1, 0x01010101u), 0xFDFDFDFDu);
      const int blk = t >> 4;
      if ((lane & 15) == 0) {
        ebw[x * 16 + 2 * blk] = pk0;
        ebw[x * 16 + 2 * blk + 1] = pk1;
      }
      // P'[(blk, g)][t] = w 2^(127 - E) in FP16 (K-major SW128: 64-key atoms, row = 8 blk + g)
      const uint32_t pt = base + OFF_P + x * P_TILE + (t >> 6) * P_ATOM;
      const int kc = t & 63;
#pragma unroll
      for (int g = 0; g < 8; g++) {
        const uint32_t e = ((g < 4 ? pk0 : pk1) >> (8 * (g & 3))) & 0xFFu;
        const __half hv = __float2half_rn(wv[g] * __uint_as_float((254u - e) << 23));
        const uint32_t addr = pt + sw128(blk * 8 + g, kc >> 3) + (kc & 7) * 2;
        asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(__half_as_ushort(hv)) : "memory");
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(bar(B_PFULL + x));
      done = i + 1;
      // fold the previous tile (its exponents were published before this tile's barrier)
      if (i >= 1) ok = fold(i - 1);
#pragma unroll
      for (int g = 0; g < 8; g++) alpha_prev[g] = alpha[g];
    }
    // final vote: the last tile's exponents become visible at this barrier too
    if (lane == 0) vote[8 + wi] = (ok && done == nT) ? 1 : 0;
    named_bar_sync(1, 128);
    const bool all_ok = vote[8] && vote[9] && vote[10] && vote[11];
    if (all_ok) fold(nT - 1);

    // ---- partial (m, l, O) of this slice per query head; thread t = d ----
#pragma unroll
    for (int g = 0; g < 8; g++)
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) lsum[g] += __shfl_xor_sync(0xffffffffu, lsum[g], off);
    if (lane == 0)
#pragma unroll
      for (int g = 0; g < 8; g++) lred[wi * 8 + g] = lsum[g];
    named_bar_sync(1, 128);
    for (int g = 0; g < G; g++) {
      const int64_t prow = ((row0 * a.num_q_heads) + h * G + g) * a.num_splits + split;
      a.part_acc[prow * kHeadDim + t] = O[g];
      if (t == 0) {
        a.part_ml[prow * 2] = m[g];
        a.part_ml[prow * 2 + 1] = lred[g] + lred[8 + g] + lred[16 + g] + lred[24 + g];
      }
    }
  }

  // ======================= teardown, then the merge by the last slice to arrive =======================
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
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
  float* wts = reinterpret_cast<float*>(gbase);  // the gather ring is idle now
  for (int i = threadIdx.x; i < G * nslices; i += blockDim.x) {
    const int g = i / nslices, sl = i % nslices;
    const int64_t prow = ((row0 * a.num_q_heads) + h * G + g) * a.num_splits + sl;
    wts[i] = __ldcg(a.part_ml + prow * 2);
    wts[G * nslices + i] = __ldcg(a.part_ml + prow * 2 + 1);
  }
  __syncthreads();
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    float* wm = wts + g * nslices;
    const float* wl = wts + G * nslices + g * nslices;
    float M = -INFINITY;
    for (int sl = 0; sl < nslices; sl++) M = fmaxf(M, wm[sl]);
    float L = 0.0f;
    if (M != -INFINITY)
      for (int sl = 0; sl < nslices; sl++) L += exp2f(wm[sl] - M) * wl[sl];
    const float invL = (M != -INFINITY && L > 0.0f) ? 1.0f / L : 0.0f;
    for (int sl = 0; sl < nslices; sl++) wm[sl] = (invL != 0.0f) ? exp2f(wm[sl] - M) * invL : 0.0f;
  }
  __syncthreads();
  for (int it = threadIdx.x; it < G * (kHeadDim / 4); it += blockDim.x) {
    const int d4 = it % (kHeadDim / 4), g = it / (kHeadDim / 4);
    const int64_t basep = ((row0 * a.num_q_heads) + h * G + g) * a.num_splits;
    const float* wm = wts + g * nslices;
    const float4* src = reinterpret_cast<const float4*>(a.part_acc + basep * kHeadDim) + d4;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    int sl = 0;
    for (; sl + 8 <= nslices; sl += 8) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; u++) v[u] = __ldcg(src + static_cast<int64_t>(sl + u) * (kHeadDim / 4));
#pragma unroll
      for (int u = 0; u < 8; u++) {
        const float wv = wm[sl + u];
        o.x += wv * v[u].x;
        o.y += wv * v[u].y;
        o.z += wv * v[u].z;
        o.w += wv * v[u].w;
      }
    }
    for (; sl < nslices; sl++) {
      const float4 v = __ldcg(src + static_cast<int64_t>(sl) * (kHeadDim / 4));
      const float wv = wm[sl];
      o.x += wv * v.x;
      o.y += wv * v.y;
      o.z += wv * v.z;
      o.w += wv * v.w;
    }
    const uint2 packed = make_uint2(float2_to_bf16x2(o.x, o.y), float2_to_bf16x2(o.z, o.w));
    *reinterpret_cast<uint2*>(a.out + (row0 * a.num_q_heads + h * G + g) * kHeadDim + 4 * d4) = packed;
  }
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
  decode_tc_kernel<<<grid, 320, SMEM_ALLOC, s>>>(tmk, tmv, a);
  return cudaGetLastError();
}

}  // namespace ftkv
