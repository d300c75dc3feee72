// decode_tok.cu -- split-K decode attention for single-row batches, token-major loads.
//
// What it computes is what decode.cu computes (FreeToken PR #897, opening description and "Fresh R9700
// stage-1 A/B"): for a request with n keys and a BF16 query row, per query head i (KV head h = i / G)
//     s_j = (q . k^_j) * sm_scale,   k^_j = decode(codeK_j) * scaleK_j,   v^_j likewise,
//     o   = sum_j softmax(s)_j v^_j,
// with split-K over the keys and the split merge in the same call.  Per 16-key block, QK^T runs on the
// FP8 tensor cores on the stored codes (the query in two exact E4M3 pieces) and PV on FP16 tensor cores on
// the exactly converted V codes.
//
// Head dimension D = 128, or 256 (the full-attention layers of FreeToken's Qwen3.6 case, PR #897 "Known
// regression and uncertainty"): a 256-d head is two 128-d halves, each loaded, multiplied and accumulated
// like a 128-d head; the 256-d kernel runs one CTA per SM (its ring alone takes ~198 KB, and each lane holds
// 64 accumulators).
//
// The unit of work and of memory traffic:
//  * A CTA covers one key slice of a request for HC (up to 4) KV heads at once.  The codes of one token
//    for those heads are one contiguous run of HC x D bytes in the pool ([rows][Hkv][D]), and a warp
//    loads whole runs with one 16-byte cp.async per lane.  Random 512-byte runs stream from HBM at about
//    1.5x the rate of random 128-byte rows (the rows of one token read by four different CTAs).
//  * Warps form NG = 8 / HC key groups of HC warps, one warp per KV head.  A group shares a 3-stage ring
//    of 16-key blocks (K and V runs of all HC heads plus their scales); the HC warps of a group load a
//    block together and meet at a named barrier before computing it.  At the end the groups' partials
//    (m, l, accumulator) are combined in shared memory, so a key slice yields one partial per query head,
//    written transposed (one quad of d over the slices is contiguous) for the merge's loads.
//  * The split merge: when the grid fits on the GPU at once (batch 1), a cooperative launch, a grid barrier
//    and the merge spread over the whole grid (coop_finish); otherwise a second small kernel behind this
//    one (decode_merge_kernel).
//  * (D = 128) 112 KB of shared memory and 8 warps of at most 128 registers: two CTAs fit on one SM, so the CTAs
//    of the next decode launch in the stream (programmatic dependent launch) become resident while this
//    launch's CTAs still run.  With FTKV_DECODE_STABLE_HISTORY (the caller guarantees that no pending
//    work writes the slot table, the sequence lengths or the history rows), a CTA fills its whole ring
//    with history blocks before waiting for the preceding grid, so its loads overlap the tail of the
//    previous launch (the grid barrier and the merge).  The query, the new tokens and everything written
//    are touched only after the wait.
//  * The scale of a row is 4 bytes at a random place: a gather of one is a whole DRAM access for one
//    sector.  When the keys may cover most of the pool (batch 1 at long context), every CTA first
//    requests its share of both scale arrays into L2 with one bulk prefetch each (a hint, issued before
//    the wait), and the per-key scale reads then hit L2.
//
// (Loading each key's run with one bulk copy (cp.async.bulk, 512 B, completion on a per-stage mbarrier,
// issued by one warp per group) instead of 16-byte cp.async by every lane measured slower on the 48-layer
// 32K step: 831 us against 692 us -- hundreds of small copies per SM and layer; so did an L2 bulk prefetch of
// each key's runs two blocks ahead of the ring: 848 us against 688 us.)
//
// Per-block arithmetic is kept short, because at batch 1 the block loop is bound by instruction issue,
// not by memory:
//  * the softmax maximum is lazy: the running maximum m (log2 units) is raised, and the accumulator
//    rescaled, only when a score exceeds it by more than 8 (a warp vote; otherwise p = 2^(s - m) <= 2^8);
//  * PV accumulates in place.  The value-weighted probabilities w_j = p_j * scaleV_j enter the FP16 MMA as
//    w_j * 2^-E, with one power-of-two exponent E per query head that only grows: it is raised (and the
//    accumulator rescaled exactly by a power of two) when some w_j would exceed 2^(E+12), so every FP16
//    operand stays below 2^13.  FP16 has a narrow exponent range and the per-row V scales of a slice can
//    span 2^30; terms far below the largest ones lose FP16 precision only in proportion to their share
//    of the sum.
//  * The new token of a fused store is quantized once into shared memory and patched into its block,
//    instead of being written, fenced and read back.
#include <cfloat>
#include <mutex>

#include "decode_common.cuh"
#include "decode_merge.cuh"
#include "ftkv_device.cuh"
#include "ftkv_internal.h"

namespace ftkv {
namespace {

constexpr int TW = 8;      // warps per CTA
constexpr int TKB = 16;    // keys per block
constexpr int TNS = 3;     // ring stages per key group
constexpr int TWIN = 1024; // slot indices staged in shared memory at a time
constexpr float kLazyMax = 8.0f;   // log2 slack of the running maximum
constexpr int kLazyExp = 12;       // w may reach 2^(E + kLazyExp) before E is raised

// HC KV heads per CTA, head dimension D (128 or 256).
template <int HC, int D>
struct Tok {
  static constexpr int NG = TW / HC;                      // key groups
  static constexpr int RUN = HC * D;                      // bytes of one token's codes for the HC heads
  static constexpr int V_OFF = TKB * RUN;                 // stage: K runs [16][RUN], V runs [16][RUN],
  static constexpr int S_OFF = 2 * TKB * RUN;             //        K scales [16][HC], V scales [16][HC]
  static constexpr int STAGE = 2 * TKB * RUN + 2 * TKB * HC * 4;
  static constexpr int RING = NG * TNS * STAGE;
  static constexpr int SLOT_OFF = RING;                   // [TWIN] int32 slot indices
  static constexpr int NEW_OFF = SLOT_OFF + TWIN * 4;     // new token: [HC][K D | V D] codes, [HC][2] scales
  static constexpr int SMEM = NEW_OFF + HC * (2 * D + 8);
  static constexpr int CTAS_PER_SM = D == 128 ? 2 : 1;    // D = 256: the ring alone takes ~198 KB
  static constexpr int KSTEP = 512 / D;                   // keys whose runs one load round covers
  static constexpr int NSW = 8 / KSTEP;                   // load rounds before the swizzle pattern repeats
};
static_assert(Tok<4, 128>::SMEM <= 113 * 1024 && Tok<2, 128>::SMEM <= 113 * 1024 && Tok<1, 128>::SMEM <= 113 * 1024,
              "two CTAs per SM");
static_assert(Tok<4, 256>::SMEM <= 227 * 1024 && Tok<2, 256>::SMEM <= 227 * 1024 && Tok<1, 256>::SMEM <= 227 * 1024,
              "one CTA per SM");

// Shared-memory offsets of 16-byte chunk p of KV head hd of key `key` within a stage.  K is read as
// (key g, chunks 2t and 2t+1 of each 128-d half) and V as (keys 2t.., chunk g of each half); the XOR swizzles
// (on the chunk's low three bits) keep both reads and the run-wide cp.async writes free of bank conflicts.
template <int HC, int D>
__device__ __forceinline__ uint32_t tk_off(int key, int hd, int p) {
  return key * Tok<HC, D>::RUN + hd * D + ((p ^ (key & 7)) << 4);
}
template <int HC, int D>
__device__ __forceinline__ uint32_t tv_off(int key, int hd, int p) {
  return Tok<HC, D>::V_OFF + key * Tok<HC, D>::RUN + hd * D + ((p ^ (((key >> 1) & 3) << 1)) << 4);
}

template <int HC, int D>
__global__ void __launch_bounds__(TW * 32, Tok<HC, D>::CTAS_PER_SM) decode_tok_kernel(const DecodeArgs a) {
  using T = Tok<HC, D>;
  constexpr int NH = D / 128;  // 128-d halves
  constexpr int NG = T::NG;
  extern __shared__ __align__(128) uint8_t smem[];
  int32_t* sslot = reinterpret_cast<int32_t*>(smem + T::SLOT_OFF);
  uint8_t* newtok = smem + T::NEW_OFF;

  const int split = blockIdx.x, b = blockIdx.z;
  const int h0 = blockIdx.y * HC;  // first KV head of this CTA
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int gi = warp / HC, hh = warp % HC;          // key group, KV head within the CTA
  const int lt = threadIdx.x - gi * 32 * HC;         // thread within the key group
  const int64_t hkv = a.num_kv_heads;
  const int64_t tok_stride = hkv * D;                // bytes between consecutive pool rows' codes

  griddep_launch_dependents();
  if (a.scan_scales && threadIdx.x < 2) {  // this CTA's share of the K (thread 0) and V (thread 1) scale array
    const int ncta = gridDim.x * gridDim.y * gridDim.z;
    const int cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    const int64_t total = a.num_rows * hkv * 4;           // bytes of one scale array
    const int64_t share = ((total + ncta - 1) / ncta + 15) / 16 * 16;
    const int64_t lo = share * cta;
    const int64_t hi = (lo + share < total) ? lo + share : total;
    // whole 16-byte aligned units inside [base + lo, base + hi) (the array itself need only be 4-byte aligned)
    const uintptr_t base = reinterpret_cast<uintptr_t>(threadIdx.x ? a.v_scales : a.k_scales);
    const uintptr_t p0 = (base + lo + 15) & ~uintptr_t(15), p1 = (base + hi) & ~uintptr_t(15);
    if (p1 > p0) prefetch_l2_bulk(reinterpret_cast<const void*>(p0), static_cast<uint32_t>(p1 - p0));
  }
  const bool early = a.early != 0;
  if (!early) griddep_wait();

  // ---- slice geometry (seq_lens and the slot table are stable before the wait under the contract) ----
  const int64_t n = clamp_seq_len(a, b, threadIdx.x == 0 && split == 0 && blockIdx.y == 0);
  // slices cover keys [first, n): first = 0, or n - W with a sliding window (one query row per request)
  const int j0 = static_cast<int>(first_key(a, n, 1)) + split * static_cast<int>(a.chunk);  // 32-bit (host check)
  const int j1 = (static_cast<int64_t>(j0) + a.chunk < n) ? j0 + static_cast<int>(a.chunk) : static_cast<int>(n);
  const bool has_keys = j0 < j1;
  const int hist_end = static_cast<int>(n) - a.max_q_rows;  // keys below are history (never written here)
  const int new_pos = a.k_new ? static_cast<int>(n) - 1 : -1;  // the fused store's token, if any
  const uint32_t ring = smem_addr(smem) + gi * TNS * T::STAGE;

  // ---- per-thread load plan: every block, this thread copies 16 bytes of the K run and of the V run of
  // keys kb, kb + KSTEP, .. (16 / KSTEP keys; chunk `rem` of the HC-head run), and one scale ----
  constexpr int KSTEP = T::KSTEP, NSW = T::NSW, CPH = D / 16;  // CPH: 16-byte chunks per head row
  const int kb = lt / (CPH * HC), rem = lt % (CPH * HC);
  const int ld_hd = rem / CPH, ld_p = rem % CPH;
  uint32_t dko[NSW], dvo[NSW];  // the swizzled destinations of keys kb + r KSTEP repeat every 8 keys
#pragma unroll
  for (int r = 0; r < NSW; r++) {
    dko[r] = tk_off<HC, D>(kb + r * KSTEP, ld_hd, ld_p);
    dvo[r] = tv_off<HC, D>(kb + r * KSTEP, ld_hd, ld_p);
  }
  const int64_t goff = h0 * D + rem * 16;
  const int s_sel = lt / (TKB * HC), s_idx = lt % (TKB * HC);   // scale: tensor, (key, head) index
  const int s_key = s_idx / HC, s_hd = s_idx % HC;
  const float* s_base = (s_sel ? a.v_scales : a.k_scales) + h0 + s_hd;
  const uint32_t s_dst = T::S_OFF + (s_sel * TKB * HC + s_idx) * 4;
  const uint64_t pol = l2_policy_evict_first();  // the key loop reads every line once

  auto stage_slots = [&](int js, int nk) {
    for (int i = threadIdx.x; i < nk; i += blockDim.x) {
      int32_t sv = a.req_to_slot[static_cast<int64_t>(b) * a.req_stride + js + i];
      if (sv < 0 || sv >= a.num_rows) {
        flag_error(a.err, kDevErrBadSlot);
        sv = 0;
      }
      sslot[i] = sv;
    }
  };
  // Block i of this group within the window [js, js + nk): keys js + (gi + i NG) 16 .. +15, into stage
  // i % TNS.  Keys past the window are zero-filled; the fused store's token is not loaded (it is patched
  // in from shared memory before the block is computed).
  auto issue = [&](int i, int my_nblk, int js, int nk) {
    if (i < my_nblk) {
      const int key0 = (gi + i * NG) * TKB;
      const uint32_t st = ring + (i % TNS) * T::STAGE;
#pragma unroll
      for (int r = 0; r < TKB / KSTEP; r++) {
        const int key = key0 + kb + r * KSTEP;
        const uint32_t dk = st + dko[r % NSW] + (r / NSW) * 8 * T::RUN;
        const uint32_t dv = st + dvo[r % NSW] + (r / NSW) * 8 * T::RUN;
        if (key < nk) {
          if (js + key != new_pos) {
            const int64_t off = static_cast<int64_t>(sslot[key]) * tok_stride + goff;
            cp_async_16_hint(dk, a.k_codes + off, pol);
            cp_async_16_hint(dv, a.v_codes + off, pol);
          }
        } else {
          st_shared_zero16(dk);
          st_shared_zero16(dv);
        }
      }
      const int key = key0 + s_key;
      if (key < nk) {
        if (js + key != new_pos) cp_async_4(st + s_dst, s_base + static_cast<int64_t>(sslot[key]) * hkv);
      } else {
        st_shared_u32(st + s_dst, 0u);
      }
    }
    cp_async_commit();
  };
  auto window_blocks = [&](int nk) {  // this group's blocks in a window of nk keys
    const int nblk = (nk + TKB - 1) / TKB;
    return nblk > gi ? (nblk - gi + NG - 1) / NG : 0;
  };

  // ---- before the wait (contract): first slot window and as many history blocks as the ring holds.  (An L2
  // prefetch of the rest of the window's history here measured slower on the 48-layer 32K step: 711 us issued
  // at once, 706 us gated on the preceding launch's barrier, against 689 us without; so did triggering the next
  // launch only after the key loop, 719 us.) ----
  const int nk0 = has_keys ? ((j1 - j0 < TWIN) ? j1 - j0 : TWIN) : 0;
  int pre = 0;  // blocks of window 0 already issued (a prefix of this group's blocks)
  if (early) {
    if (has_keys) stage_slots(j0, nk0);
    __syncthreads();
    const int mb0 = window_blocks(nk0);
    for (int i = 0; i < TNS; i++) {  // group-uniform
      const int blk_end = j0 + (gi + i * NG) * TKB + TKB;
      if (i >= mb0 || blk_end > hist_end) break;
      issue(i, mb0, j0, nk0);
      pre = i + 1;
    }
    {
      // the query rows of the CTA's heads (written by the preceding work in a model, so usually in L2
      // already; a prefetch is a hint and reads nothing)
      if (!a.q_row_offsets && threadIdx.x < HC * a.group * 2 * NH)
        prefetch_l2_keep(a.q + (static_cast<int64_t>(b) * a.num_q_heads + h0 * a.group) * D + threadIdx.x * 64);
    }
    griddep_wait();
  }

  // ---- request rows (single-row kernel: R is 0 or 1) ----
  int64_t row0;
  int R;
  if (a.q_row_offsets) {
    row0 = a.q_row_offsets[b];
    R = a.q_row_offsets[b + 1] - a.q_row_offsets[b];
  } else {
    row0 = b;
    R = 1;
  }
  const bool bad_rows = R < 0 || R > a.max_q_rows || row0 < 0 || row0 + R > a.total_q_rows;
  if (bad_rows || !has_keys || R == 0) {  // nothing to publish (the merge writes zeros where needed)
    if (bad_rows && threadIdx.x == 0 && split == 0 && blockIdx.y == 0) flag_error(a.err, kDevErrQRows);
    cp_async_wait<0>();  // nothing in flight when the CTA leaves
    if (a.coop) coop_finish<TW>(a);
    return;
  }

  if (!early) stage_slots(j0, nk0);

  // ---- query loads: each warp its own KV head's query heads; lane (g, t) takes d = 128hf + 32t .. +31 of
  // query head g (every load in flight at once) ----
  const int G = a.group;
  const bool qok = g < G;  // heads past the group pad the 8-wide MMA N dimension with zeros
  uint4 qr[NH][4];
  {
    const uint4* qsrc = reinterpret_cast<const uint4*>(a.q + (row0 * a.num_q_heads + (h0 + hh) * G + (qok ? g : 0)) * D);
#pragma unroll
    for (int hf = 0; hf < NH; hf++)
#pragma unroll
      for (int c = 0; c < 4; c++) qr[hf][c] = qok ? __ldg(qsrc + 16 * hf + 4 * t + c) : make_uint4(0u, 0u, 0u, 0u);
  }

  // ---- fused store of the request's new token (position n - 1), if it falls in this slice: one warp per
  // KV head, K row on lanes 0-15 and V row on lanes 16-31, with the store kernel's arithmetic; the codes and
  // scales also go to shared memory, from where they are patched into the token's block ----
  const bool has_new = new_pos >= j0 && new_pos < j1;  // CTA-uniform (R == 1 here)
  // (D = 256: one warp per (KV head, tensor), 32 lanes x 8 elements)
  constexpr int LPR = D / 8;  // lanes per row
  if (has_new && warp < HC * NH) {
    const int hd = (NH == 1) ? warp : warp >> 1;
    const int half = (NH == 1) ? lane >> 4 : warp & 1, l = lane % LPR;
    const uint16_t* src = (half ? a.v_new : a.k_new) + (row0 * hkv + h0 + hd) * D + l * 8;
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src));
    const int32_t sv = a.req_to_slot[static_cast<int64_t>(b) * a.req_stride + new_pos];
    float sc;
    const uint2 packed = quantize_row_lane8<LPR>(raw, sc);
    *reinterpret_cast<uint2*>(newtok + hd * 2 * D + half * D + l * 8) = packed;
    if (l == 0) reinterpret_cast<float*>(newtok + HC * 2 * D)[hd * 2 + half] = sc;
    if (sv >= 0 && sv < a.num_rows) {  // a bad slot is flagged when staged; nothing is written
      const int64_t row = static_cast<int64_t>(sv) * hkv + h0 + hd;
      // the pool is the caller's writable memory (ftkv_pool holds non-const pointers); later kernels see
      // these rows once this one has completed, and this kernel reads the token from shared memory
      *reinterpret_cast<uint2*>(const_cast<uint8_t*>(half ? a.v_codes : a.k_codes) + row * D + l * 8) = packed;
      if (l == 0) const_cast<float*>(half ? a.v_scales : a.k_scales)[row] = sc;
    }
  }

  // ---- query pieces: x = q * 2^(7-ex), ex the exponent of max|q| over the head: |x| < 256; pieces
  // x = h1 + h2/16, both E4M3 (exact unless |q| < 2^-13 max|q|); multiplier 2^(ex-7) * sm_scale * log2(e).
  // They are the B operand of QK^T: query head g, d = 128hf + 32t + 8kk' + {0..3} (b0) / {4..7} (b1) for
  // k-step kk = 4hf + kk'.  The head's max comes from the 4 lanes that hold it; lane (g, t) then takes the
  // multipliers of query heads 2t, 2t+1 (its accumulator columns) from the lanes of those heads. ----
  uint32_t qp[2][4 * NH][2];
  float fq[2];
  {
    float amax = 0.0f;
#pragma unroll
    for (int hf = 0; hf < NH; hf++)
#pragma unroll
      for (int c = 0; c < 4; c++) {
        const uint4 w = qr[hf][c];
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(w.x)), fabsf(bf16_hi(w.x))), fmaxf(fabsf(bf16_lo(w.y)), fabsf(bf16_hi(w.y)))));
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(w.z)), fabsf(bf16_hi(w.z))), fmaxf(fabsf(bf16_lo(w.w)), fabsf(bf16_hi(w.w)))));
      }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    int ex = (amax > 0.0f) ? ilogbf(amax) : 0;
    ex = ex < -120 ? -120 : ex;
    const float up = __uint_as_float(static_cast<uint32_t>(127 + 7 - ex) << 23);
    auto pieces4 = [&](uint32_t w01, uint32_t w23, uint32_t& p0, uint32_t& p1) {  // 4 elements -> 2 words
      float x0 = bf16_lo(w01) * up, x1 = bf16_hi(w01) * up, x2 = bf16_lo(w23) * up, x3 = bf16_hi(w23) * up;
      const uint32_t c01 = e4m3x2_encode(x0, x1), c23 = e4m3x2_encode(x2, x3);
      p0 = c01 | (c23 << 16);
      const float2 v01 = f16x2_to_float2(e4m3x2_to_f16x2(c01));
      const float2 v23 = f16x2_to_float2(e4m3x2_to_f16x2(c23));
      x0 = (x0 - v01.x) * 16.0f;
      x1 = (x1 - v01.y) * 16.0f;
      x2 = (x2 - v23.x) * 16.0f;
      x3 = (x3 - v23.y) * 16.0f;
      p1 = e4m3x2_encode(x0, x1) | (e4m3x2_encode(x2, x3) << 16);
    };
#pragma unroll
    for (int hf = 0; hf < NH; hf++)
#pragma unroll
      for (int c = 0; c < 4; c++) {
        const uint4 w = qr[hf][c];
        pieces4(w.x, w.y, qp[0][4 * hf + c][0], qp[1][4 * hf + c][0]);
        pieces4(w.z, w.w, qp[0][4 * hf + c][1], qp[1][4 * hf + c][1]);
      }
    const float mult = __uint_as_float(static_cast<uint32_t>(127 - 7 + ex) << 23) * a.qk_scale_log2;
    fq[0] = __shfl_sync(0xffffffffu, mult, (2 * t) * 4);
    fq[1] = __shfl_sync(0xffffffffu, mult, (2 * t + 1) * 4);
  }
  if (!early || has_new) __syncthreads();  // the staged slots (after the wait) and the new token's codes
  // fragment offsets within a stage (loop-invariant)
  // (the second 128-d half: chunks 8 + the first half's, same swizzle; tk_off(key, hd, p + 8) = that + 128)
  const uint32_t oK0 = tk_off<HC, D>(g, hh, 2 * t), oK1 = tk_off<HC, D>(g, hh, 2 * t + 1);
  const uint32_t oK2 = tk_off<HC, D>(g + 8, hh, 2 * t), oK3 = tk_off<HC, D>(g + 8, hh, 2 * t + 1);
  const uint32_t oV0 = tv_off<HC, D>(2 * t, hh, g), oV1 = tv_off<HC, D>(2 * t + 1, hh, g);
  const uint32_t oV2 = tv_off<HC, D>(2 * t + 8, hh, g), oV3 = tv_off<HC, D>(2 * t + 9, hh, g);
  const uint32_t oS0 = T::S_OFF + (g * HC + hh) * 4, oS1 = T::S_OFF + ((g + 8) * HC + hh) * 4;
  constexpr uint32_t VS = TKB * HC * 4;  // V scales follow the K scales

  constexpr int MT = D / 16;  // accumulator tiles: d = 128hf + 16g + ..
  float acc[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; mt++) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.0f;
  float m[2] = {-INFINITY, -INFINITY};  // running maximum of s (log2 units), per query head 2t, 2t+1
  float l[2] = {0.0f, 0.0f};            // this lane's share of sum 2^(s - m)
  int E[2] = {-126, -126};              // FP16 operand exponent: PV takes w * 2^-E
  float wlim[2] = {exp2i(-126 + kLazyExp), exp2i(-126 + kLazyExp)};
  float iw[2] = {exp2i(126), exp2i(126)};

  for (int js = j0; js < j1; js += TWIN) {  // CTA-uniform
    const int je = (js + TWIN < j1) ? js + TWIN : j1;
    const int nk = je - js;
    int done = 0;  // blocks of this window already issued
    if (js == j0) {
      done = pre;
    } else {
      __syncthreads();  // every group is done with the previous window's slots and stages
      stage_slots(js, nk);
      __syncthreads();
    }
    const int my_nblk = window_blocks(nk);
    for (int i = done; i < TNS; i++) issue(i, my_nblk, js, nk);  // the rest of the prologue: TNS groups
    const int new_key = (has_new && new_pos >= js && new_pos < je) ? new_pos - js : -1;  // window-relative

#pragma unroll 1
    for (int i = 0; i < my_nblk; i++) {
      if (i == 0) cp_async_wait<TNS - 1>(); else cp_async_wait<TNS - 2>();
      group_barrier<NG>(gi, 32 * HC);  // every copy of block i landed; every warp is done with block i - 1
      const uint32_t st = ring + (i % TNS) * T::STAGE;
      const int key0 = (gi + i * NG) * TKB;
      if (new_key >= key0 && new_key < key0 + TKB) {  // warp-uniform: patch this head's new token in
        const int kk = new_key - key0;
        const uint8_t* nt = newtok + hh * 2 * D;
        if (lane < CPH)
          st_shared_v4(st + tk_off<HC, D>(kk, hh, lane), *reinterpret_cast<const uint4*>(nt + lane * 16));
        else if (lane < 2 * CPH)
          st_shared_v4(st + tv_off<HC, D>(kk, hh, lane - CPH), *reinterpret_cast<const uint4*>(nt + D + (lane - CPH) * 16));
        if (lane < 2)
          st_shared_u32(st + T::S_OFF + lane * VS + (kk * HC + hh) * 4,
                        __float_as_uint(reinterpret_cast<const float*>(newtok + HC * 2 * D)[hh * 2 + lane]));
        __syncwarp();
      }
      const int jb = js + key0;

      // ---- S^T = K Q^T on E4M3 codes: keys as M (rows g, g+8), query heads as N, 2 query pieces ----
      float c[2][4];
#pragma unroll
      for (int p = 0; p < 2; p++) c[p][0] = c[p][1] = c[p][2] = c[p][3] = 0.0f;
#pragma unroll
      for (int hf = 0; hf < NH; hf++) {
        const uint4 kA0 = ld_shared_v4(st + oK0 + 128 * hf);
        const uint4 kA1 = ld_shared_v4(st + oK1 + 128 * hf);
        const uint4 kB0 = ld_shared_v4(st + oK2 + 128 * hf);
        const uint4 kB1 = ld_shared_v4(st + oK3 + 128 * hf);
#pragma unroll
        for (int kk = 0; kk < 4; kk++) {
          const uint4& A = kk < 2 ? kA0 : kA1;
          const uint4& B = kk < 2 ? kB0 : kB1;
          const uint32_t a0 = word(A, 2 * (kk & 1)), a2 = word(A, 2 * (kk & 1) + 1);
          const uint32_t a1 = word(B, 2 * (kk & 1)), a3 = word(B, 2 * (kk & 1) + 1);
#pragma unroll
          for (int p = 0; p < 2; p++)
            mma_e4m3_16832(c[p], a0, a1, a2, a3, qp[p][4 * hf + kk][0], qp[p][4 * hf + kk][1]);
        }
      }
      const float skg = ld_shared_f32(st + oS0), skg8 = ld_shared_f32(st + oS1);
      const float svg = ld_shared_f32(st + oS0 + VS), svg8 = ld_shared_f32(st + oS1 + VS);

      // ---- softmax with a lazy maximum (log2 domain) ----
      const bool in0 = jb + g < je, in8 = jb + g + 8 < je;
      const float s0 = in0 ? fmaf(c[1][0], 1.0f / 16.0f, c[0][0]) * (skg * fq[0]) : -INFINITY;
      const float s1 = in0 ? fmaf(c[1][1], 1.0f / 16.0f, c[0][1]) * (skg * fq[1]) : -INFINITY;
      const float s2 = in8 ? fmaf(c[1][2], 1.0f / 16.0f, c[0][2]) * (skg8 * fq[0]) : -INFINITY;
      const float s3 = in8 ? fmaf(c[1][3], 1.0f / 16.0f, c[0][3]) * (skg8 * fq[1]) : -INFINITY;
      const bool raise = fmaxf(s0, s2) > m[0] + kLazyMax || fmaxf(s1, s3) > m[1] + kLazyMax;
      if (__any_sync(0xffffffffu, raise)) {  // new maximum: exact block max, rescale
        float bm0 = fmaxf(s0, s2), bm1 = fmaxf(s1, s3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
          bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
        }
        const float mn0 = fmaxf(m[0], bm0), mn1 = fmaxf(m[1], bm1);
        const float al0 = (m[0] == -INFINITY) ? 1.0f : fast_exp2(m[0] - mn0);
        const float al1 = (m[1] == -INFINITY) ? 1.0f : fast_exp2(m[1] - mn1);
        m[0] = mn0;
        m[1] = mn1;
        l[0] *= al0;
        l[1] *= al1;
#pragma unroll
        for (int mt = 0; mt < MT; mt++) {
          acc[mt][0] *= al0;
          acc[mt][1] *= al1;
          acc[mt][2] *= al0;
          acc[mt][3] *= al1;
        }
      }
      const float mu0 = (m[0] == -INFINITY) ? 0.0f : m[0], mu1 = (m[1] == -INFINITY) ? 0.0f : m[1];
      const float p0 = fast_exp2(s0 - mu0), p1 = fast_exp2(s1 - mu1);
      const float p2 = fast_exp2(s2 - mu0), p3 = fast_exp2(s3 - mu1);
      l[0] += p0 + p2;
      l[1] += p1 + p3;
      const float w0 = p0 * svg, w1 = p1 * svg, w2 = p2 * svg8, w3 = p3 * svg8;
      // ---- lazy FP16 exponent: raise E (rescaling by an exact power of two) when some w would exceed
      // 2^(E + kLazyExp) ----
      const bool grow = fmaxf(w0, w2) > wlim[0] || fmaxf(w1, w3) > wlim[1];
      if (__any_sync(0xffffffffu, grow)) {
        float W0 = fmaxf(w0, w2), W1 = fmaxf(w1, w3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          W0 = fmaxf(W0, __shfl_xor_sync(0xffffffffu, W0, off));
          W1 = fmaxf(W1, __shfl_xor_sync(0xffffffffu, W1, off));
        }
        // exponent of W (a subnormal W counts as -126); E never decreases
        const int e0 = max(E[0], max(static_cast<int>(__float_as_uint(W0) >> 23), 1) - 127);
        const int e1 = max(E[1], max(static_cast<int>(__float_as_uint(W1) >> 23), 1) - 127);
        const int ne0 = min(e0, 127 - kLazyExp), ne1 = min(e1, 127 - kLazyExp);
        // <= 1, exact (0 below 2^-126: the earlier terms vanish next to the new ones)
        const float f0 = (E[0] - ne0 < -126) ? 0.0f : exp2i(E[0] - ne0);
        const float f1 = (E[1] - ne1 < -126) ? 0.0f : exp2i(E[1] - ne1);
        E[0] = ne0;
        E[1] = ne1;
        wlim[0] = exp2i(ne0 + kLazyExp);
        wlim[1] = exp2i(ne1 + kLazyExp);
        iw[0] = exp2i(-ne0);
        iw[1] = exp2i(-ne1);
#pragma unroll
        for (int mt = 0; mt < MT; mt++) {
          acc[mt][0] *= f0;
          acc[mt][1] *= f1;
          acc[mt][2] *= f0;
          acc[mt][3] *= f1;
        }
      }
      // The copies of block i + TNS - 1 go into the stage of block i - 1 (free since the barrier).  They are issued
      // here, between the softmax and the PV product, rather than right after the barrier: a warp stalls for
      // hundreds of cycles while the SM takes in its copy requests, and here that stall overlaps less with this
      // block's shared-memory loads (48-layer 32K step: 676 us against 685 us issued after the barrier).
      if (i > 0) issue(i + TNS - 1, my_nblk, js, nk);
      const uint32_t pb0 = movmatrix_trans(float2_to_f16x2(w0 * iw[0], w1 * iw[1]));   // keys 0..7
      const uint32_t pb1 = movmatrix_trans(float2_to_f16x2(w2 * iw[0], w3 * iw[1]));   // keys 8..15

      // ---- O^T += V^T P'^T in place: d as M (tile 8hf + 2w + {0, 1}: d = 128hf + 16g + 4w + {0, 1} / {2, 3}),
      // query heads as N, keys as K ----
#pragma unroll
      for (int hf = 0; hf < NH; hf++) {
        const uint4 v0 = ld_shared_v4(st + oV0 + 128 * hf);
        const uint4 v1 = ld_shared_v4(st + oV1 + 128 * hf);
        const uint4 v8 = ld_shared_v4(st + oV2 + 128 * hf);
        const uint4 v9 = ld_shared_v4(st + oV3 + 128 * hf);
#pragma unroll
        for (int w = 0; w < 4; w++) {
          const uint32_t x0 = word(v0, w), x1 = word(v1, w), x8 = word(v8, w), x9 = word(v9, w);
          const uint32_t lo01 = prmt(x0, x1, 0x5140), hi01 = prmt(x0, x1, 0x7362);
          const uint32_t lo89 = prmt(x8, x9, 0x5140), hi89 = prmt(x8, x9, 0x7362);
          mma_f16_16816(acc[8 * hf + 2 * w], e4m3_lo2(lo01), e4m3_hi2(lo01), e4m3_lo2(lo89), e4m3_hi2(lo89), pb0, pb1);
          mma_f16_16816(acc[8 * hf + 2 * w + 1], e4m3_lo2(hi01), e4m3_hi2(hi01), e4m3_lo2(hi89), e4m3_hi2(hi89), pb0,
                        pb1);
        }
      }
    }
    cp_async_wait<0>();
  }

  // ---- one partial per (row, query head) and key slice: the NG key groups' partials are combined in shared
  // memory first (groups 1 .. NG-1 leave m, l and the accumulator, scaled to units of 2^m, in the ring area;
  // group 0 folds them into its own), then written in the transposed layout (see DecodeArgs::ptrans) ----
#pragma unroll
  for (int hx = 0; hx < 2; hx++)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) l[hx] += __shfl_xor_sync(0xffffffffu, l[hx], off);
  // lane (g, t) holds d = 128hf + 16g + 4q4 + {0..3} of query head 2t + hx: acc[8hf+2q4][hx], acc[8hf+2q4][2+hx],
  // acc[8hf+2q4+1][hx], acc[8hf+2q4+1][2+hx]; bring it to units of 2^m
#pragma unroll
  for (int hx = 0; hx < 2; hx++) {
    const float up = exp2i(E[hx]);
#pragma unroll
    for (int mt = 0; mt < MT; mt++) {
      acc[mt][hx] *= up;
      acc[mt][2 + hx] *= up;
    }
  }
  if constexpr (NG > 1) {
    float* gacc = reinterpret_cast<float*>(smem);                   // [NG-1][HC][8][D]
    float* gml = gacc + (NG - 1) * HC * 8 * D;                      // [NG-1][HC][8][2]
    __syncthreads();  // every group is done with the ring
    if (gi > 0) {
#pragma unroll
      for (int hx = 0; hx < 2; hx++) {
        const int slot = ((gi - 1) * HC + hh) * 8 + 2 * t + hx;
#pragma unroll
        for (int hf = 0; hf < NH; hf++) {
          float4* dst = reinterpret_cast<float4*>(gacc + slot * D + 128 * hf + 16 * g);
#pragma unroll
          for (int q4 = 0; q4 < 4; q4++) {
            const int mt = 8 * hf + 2 * q4;
            dst[q4] = make_float4(acc[mt][hx], acc[mt][2 + hx], acc[mt + 1][hx], acc[mt + 1][2 + hx]);
          }
        }
        if (g == 0) *reinterpret_cast<float2*>(gml + slot * 2) = make_float2(m[hx], l[hx]);
      }
    }
    __syncthreads();
#pragma unroll 1
    for (int go = 1; go < NG && gi == 0; go++) {
#pragma unroll
      for (int hx = 0; hx < 2; hx++) {
        const int slot = ((go - 1) * HC + hh) * 8 + 2 * t + hx;
        const float2 mlo = *reinterpret_cast<const float2*>(gml + slot * 2);
        const float mn = fmaxf(m[hx], mlo.x);
        if (mn == -INFINITY) continue;  // neither holds a key
        const float f = (m[hx] == -INFINITY) ? 0.0f : fast_exp2(m[hx] - mn);
        const float fo = (mlo.x == -INFINITY) ? 0.0f : fast_exp2(mlo.x - mn);
#pragma unroll
        for (int hf = 0; hf < NH; hf++) {
          const float4* src = reinterpret_cast<const float4*>(gacc + slot * D + 128 * hf + 16 * g);
#pragma unroll
          for (int q4 = 0; q4 < 4; q4++) {
            const float4 v = src[q4];
            const int mt = 8 * hf + 2 * q4;
            acc[mt][hx] = fmaf(acc[mt][hx], f, v.x * fo);
            acc[mt][2 + hx] = fmaf(acc[mt][2 + hx], f, v.y * fo);
            acc[mt + 1][hx] = fmaf(acc[mt + 1][hx], f, v.z * fo);
            acc[mt + 1][2 + hx] = fmaf(acc[mt + 1][2 + hx], f, v.w * fo);
          }
        }
        l[hx] = fmaf(l[hx], f, mlo.y * fo);
        m[hx] = mn;
      }
    }
  }
  const int64_t nsl = a.num_splits;  // one partial per slice (pps = 1)
#pragma unroll
  for (int hx = 0; hx < 2; hx++) {
    const int hq = 2 * t + hx;  // query head within the KV head's group (N column)
    if (gi == 0 && hq < G) {
      const int64_t prow = row0 * a.num_q_heads + (h0 + hh) * G + hq;
#pragma unroll
      for (int hf = 0; hf < NH; hf++) {
        float4* dst = reinterpret_cast<float4*>(a.part_acc) + (prow * (D / 4) + 32 * hf + 4 * g) * nsl + split;
#pragma unroll
        for (int q4 = 0; q4 < 4; q4++) {
          const int mt = 8 * hf + 2 * q4;
          dst[q4 * nsl] = make_float4(acc[mt][hx], acc[mt][2 + hx], acc[mt + 1][hx], acc[mt + 1][2 + hx]);
        }
      }
      if (g == 0) *reinterpret_cast<float2*>(a.part_ml + (prow * nsl + split) * 2) = make_float2(m[hx], l[hx]);
    }
  }
  if (a.coop) coop_finish<TW>(a);  // grid barrier, then the merge spread over the grid
}

template <int HC, int D>
cudaError_t launch_tok(const DecodeArgs& a, cudaStream_t s, int dev) {
  using T = Tok<HC, D>;
  static std::once_flag once[kMaxDecodeDevices];
  static cudaError_t setup_err[kMaxDecodeDevices];
  static int resident[kMaxDecodeDevices];
  std::call_once(once[dev], [&] {
    setup_err[dev] = cudaFuncSetAttribute(decode_tok_kernel<HC, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          T::SMEM);
    int coop_ok = 0, sms = 0, per_sm = 0;
    if (setup_err[dev] == cudaSuccess) setup_err[dev] = cudaDeviceGetAttribute(&coop_ok, cudaDevAttrCooperativeLaunch, dev);
    if (setup_err[dev] == cudaSuccess) setup_err[dev] = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (setup_err[dev] == cudaSuccess &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_tok_kernel<HC, D>, TW * 32, T::SMEM) !=
            cudaSuccess)
      per_sm = 0;
    resident[dev] = (coop_ok && per_sm > 0 && sms > 0) ? per_sm * sms : -1;
  });
  if (setup_err[dev] != cudaSuccess) return setup_err[dev];
  const dim3 grid(a.num_splits, a.num_kv_heads / HC, a.batch);
  DecodeArgs c = a;
  c.pps = 1;
  c.ptrans = 1;
  const int64_t ctas = int64_t(grid.x) * grid.y * grid.z;
  c.coop = (resident[dev] > 0 && ctas <= resident[dev]) ? 1 : 0;
  if (c.coop) return launch_k_coop(decode_tok_kernel<HC, D>, grid, dim3(TW * 32), T::SMEM, s, c);
  cudaError_t e = launch_k(decode_tok_kernel<HC, D>, grid, dim3(TW * 32), T::SMEM, s, c);
  if (e != cudaSuccess) return e;
  const int64_t items = a.total_q_rows * a.num_q_heads * (D / 4);
  return launch_k(decode_merge_kernel<kMergeWarps>, dim3(static_cast<unsigned>((items + kMergeWarps - 1) / kMergeWarps)),
                  dim3(kMergeWarps * 32), 0, s, c);
}

}  // namespace

int decode_tok_heads_per_cta(int num_kv_heads) {
  return (num_kv_heads % 4 == 0) ? 4 : (num_kv_heads % 2 == 0) ? 2 : 1;
}

cudaError_t launch_decode_tok(const DecodeArgs& a, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDecodeDevices) return cudaErrorInvalidDevice;
  const int hc = decode_tok_heads_per_cta(a.num_kv_heads);
  if (a.head_dim == 256) {
    switch (hc) {
      case 4: return launch_tok<4, 256>(a, s, dev);
      case 2: return launch_tok<2, 256>(a, s, dev);
      default: return launch_tok<1, 256>(a, s, dev);
    }
  }
  switch (hc) {
    case 4: return launch_tok<4, 128>(a, s, dev);
    case 2: return launch_tok<2, 128>(a, s, dev);
    default: return launch_tok<1, 128>(a, s, dev);
  }
}

}  // namespace ftkv
