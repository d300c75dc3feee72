/*
 * ftkv.h -- C ABI of libftkv.so: an FP8 (E4M3FN) per-token/per-head KV cache for BF16 attention on
 * one GB300 (sm_103a) GPU.
 *
 * The operations follow three pages about FreeToken's opt-in FP8 KV cache:
 *   [#853] FreeToken PR #853 "opt-in FP8 KV cache (R9700)"
 *   [#897] FreeToken PR #897 "perf(attention): add packed fp8 kv reads on gfx1201"
 *   [#280] FreeToken issue #280 "Feature Request: opt-in FP8 KV-cache support for long-context MoE
 *          inference"
 *
 * Row format ([#853 "What changes"], [#280 "Proof of concept"]): every physical K/V row (one token,
 * one KV head) holds head_dim E4M3FN codes, one byte each, plus its own FP32 scale.  The scale is
 * dynamic: absmax(row) / 448, and code = E4M3FN(x / scale) with round-to-nearest-even, saturating at
 * +-448 (NaN -> 0x7F).  An all-zero row stores scale 0 and codes +-0.
 *
 * Conventions for every entry point:
 *   - Pointers named as device pointers must be device memory (cudaMalloc or torch CUDA tensors) of
 *     the current device, 16-byte aligned unless stated otherwise.  BF16 tensors are passed as
 *     uint16_t bit patterns.  All tensors are dense, row-major, in the layouts stated.
 *   - The library never allocates or frees device memory; the caller owns every buffer.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are asynchronous: they
 *     validate their arguments on the host, enqueue kernels on `stream` and return.
 *   - Argument errors are reported before anything is enqueued (nothing is launched).  Conditions
 *     that only the GPU can see (a slot outside the pool, a sequence length above the declared
 *     maximum) make the kernel skip the offending row and raise a flag in a per-device error word,
 *     read and cleared with ftkv_device_errors().
 *   - Supported: head_dim == 128 (and 256 for ftkv_store_quant and single-row decode, see
 *     FTKV_HEAD_DIM_256), num_q_heads % num_kv_heads == 0 with group size 1, 2, 4 or 8 (MHA/GQA),
 *     page size 1, one GPU (TP = 1).  Anything else returns FTKV_ERR_UNSUPPORTED, the
 *     configuration-time rejection of [#853 "What changes"] and [#280 limitations].
 */
#ifndef FTKV_H_
#define FTKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FTKV_ABI_VERSION 2
#define FTKV_HEAD_DIM 128
/* The 256-d head of FreeToken's Qwen3.6 full-attention layers ([#897 "Known regression and uncertainty"]):
 * supported by ftkv_store_quant and by single-row decode (max_q_rows == 1) over the FP8 pool. */
#define FTKV_HEAD_DIM_256 256
/* Split-K cap of decode.  The pages cap their kernel at 64 slices ([#897 "Fresh R9700 stage-1 A/B"]: 64
 * scratch slots / splits, a limit of that kernel's scratch budget).  Here one slice of a single-row batch
 * covers every KV head of its keys, so a batch-1 decode needs one slice per SM (152 on a GB300): the cap is
 * 256. */
#define FTKV_MAX_SPLITS 256
/* Largest number of query rows per request in multi-row decode ([#897] opening description, #900). */
#define FTKV_MAX_Q_ROWS 8
/* Largest batch (requests per decode call): one grid dimension of the decode kernels holds the requests.
 * A larger batch -> FTKV_ERR_UNSUPPORTED (split it into several calls). */
#define FTKV_MAX_BATCH 65535

/* Decode flags.
 * FTKV_DECODE_STABLE_HISTORY: the caller guarantees that no work still pending on `stream` when the call is
 *   enqueued writes req_to_slot, seq_lens, or the pool rows of the history -- the keys at positions below
 *   seq_lens[b] - max_q_rows of every request (true between the layers of a decode step: a layer's KV cache
 *   and the slot table are not written by the work of the layers before it).  The single-row kernel may then
 *   read them, and start loading history rows, before the preceding kernel in the stream has finished
 *   (programmatic dependent launch); the query, the new tokens and every output are touched only after it.
 *   Without the flag every read waits for the preceding kernel.  The results are the same either way. */
#define FTKV_DECODE_STABLE_HISTORY 0x1u

typedef enum {
  FTKV_OK = 0,
  FTKV_ERR_INVALID = -1,      /* null pointer, negative size, inconsistent sizes               */
  FTKV_ERR_UNSUPPORTED = -2,  /* head_dim, group size or other configuration outside the scope */
  FTKV_ERR_ALIGN = -3,        /* a pointer is not 16-byte aligned                              */
  FTKV_ERR_WORKSPACE = -4,    /* decode or prefill workspace too small                         */
  FTKV_ERR_CUDA = -6          /* a CUDA call or launch failed (see ftkv_last_cuda_error)       */
} ftkv_status;

/* Bits of the per-device error word (ftkv_device_errors). */
#define FTKV_DEVERR_BAD_SLOT 0x1    /* a slot index was < 0 or >= num_rows; that row was skipped     */
#define FTKV_DEVERR_SEQ_LEN 0x2     /* a seq_len was < 0 or > max_seq_len / req_stride; clamped        */
#define FTKV_DEVERR_Q_ROWS 0x4      /* q_row_offsets inconsistent (rows > max_q_rows or past the end);
                                       that request was skipped                                       */
#define FTKV_DEVERR_TIMEOUT 0x8     /* a bounded wait inside a kernel expired (internal error); the
                                       affected outputs are unspecified                               */

/* One layer's FP8 pool.  All four arrays are device memory owned by the caller.
 *   k_codes, v_codes : uint8 [num_rows][num_kv_heads][head_dim]   E4M3FN codes
 *   k_scales, v_scales: float [num_rows][num_kv_heads]            FP32 per-row scales          */
typedef struct ftkv_pool {
  uint8_t* k_codes;
  uint8_t* v_codes;
  float* k_scales;
  float* v_scales;
  int64_t num_rows;
  int32_t num_kv_heads;
  int32_t head_dim;
} ftkv_pool;

/* ---------------------------------------------------------------------------------------------
 * Quantize-on-write ([#853 "What changes"], [#853 "Follow-up model/workload search"]: every new
 * K/V row is quantized when it is written to its slot).
 *   k, v    : device BF16 [num_tokens][num_kv_heads][head_dim]
 *   slots   : device int32 [num_tokens]; token t is written to pool row slots[t].  Slots must be
 *             distinct within one call (duplicates leave one of the writers' rows, unspecified which).
 * Writes codes and scales of rows slots[0..num_tokens) of both K and V.  num_tokens == 0 is a no-op.
 * --------------------------------------------------------------------------------------------- */
int ftkv_store_quant(const ftkv_pool* pool, const uint16_t* k, const uint16_t* v,
                     const int32_t* slots, int64_t num_tokens, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Reconstruct historical rows into the shared BF16 workspace ([#853 "What changes"]: once per
 * layer, historical FP8 rows are rebuilt into one shared BF16 workspace for prefill).
 *   slots        : device int32 [num_prefix]; logical token i lives in pool row slots[i]
 *   ws_k, ws_v   : device BF16 [num_prefix][num_kv_heads][head_dim], written in logical order:
 *                  ws[i][h][d] = bf16_rne(float(decode(code[slots[i]][h][d])) * scale[slots[i]][h])
 * Bit-exact: one FP32 product, round-to-nearest-even.  num_prefix == 0 is a no-op.
 * --------------------------------------------------------------------------------------------- */
int ftkv_reconstruct_bf16(const ftkv_pool* pool, const int32_t* slots, int64_t num_prefix,
                          uint16_t* ws_k, uint16_t* ws_v, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Split-K decode attention over the FP8 pool ([#897 "Fresh R9700 stage-1 A/B"]: a stage over slices
 * of the keys followed by a merge; [#897] opening description: BF16 query, D128, GQA 4/8, per-row
 * scales; multi-row decode of up to 8 query rows per request).  One kernel launch: when the grid fits on
 * the GPU at once, every slice publishes its partial, the slices meet at a grid barrier and the merge is
 * spread over the whole grid; otherwise the last slice of each (request, KV head group) to finish merges.
 * Single-row batches (max_q_rows == 1) run a kernel whose CTAs cover every KV head of their keys (token-
 * contiguous loads); multi-row batches a kernel with one KV head per CTA.
 *
 *   q              : device BF16 [total_q_rows][num_q_heads][head_dim]; head_dim is the pool's (128, or
 *                    256 with max_q_rows == 1, else FTKV_ERR_UNSUPPORTED)
 *   req_to_slot    : device int32 [batch][req_stride]; key j of request b lives in pool row
 *                    req_to_slot[b * req_stride + j]
 *   seq_lens       : device int32 [batch]; request b attends to keys 0 .. seq_lens[b]-1 (the keys of
 *                    its new rows included; they must already be stored)
 *   q_row_offsets  : device int32 [batch + 1]; request b owns query rows
 *                    [q_row_offsets[b], q_row_offsets[b+1]), at most FTKV_MAX_Q_ROWS of them.  Row r
 *                    of R sees keys 0 .. seq_lens[b] - R + r (causal within the new rows).  NULL means
 *                    one row per request (total_q_rows == batch).
 *   max_q_rows     : host upper bound on rows per request (1 .. FTKV_MAX_Q_ROWS)
 *   max_seq_len    : host upper bound on seq_lens (<= req_stride); it fixes the split geometry
 *   sm_scale       : softmax scale (1/sqrt(head_dim) for the standard case)
 *   window         : 0 = full attention; W >= 1 = sliding window: a row that sees keys 0 .. v-1 attends
 *                    only to keys max(0, v - W) .. v - 1 (the "odd sliding window" integration case of
 *                    [#897 "Regression and CUDA isolation"]); the key slices then cover only the last
 *                    W + R - 1 keys of each request.  window < 0 -> FTKV_ERR_INVALID.
 *   num_splits     : 0 = automatic (fills the SMs), else 1 .. FTKV_MAX_SPLITS key slices per request
 *                    (over the window's keys when window > 0)
 *   flags          : 0 or FTKV_DECODE_STABLE_HISTORY (see above); other bits -> FTKV_ERR_INVALID
 *   workspace      : device scratch of at least ftkv_decode_workspace_bytes(...) bytes, 256-byte
 *                    aligned, ZERO-FILLED before its first use (e.g. cudaMemsetAsync).  It holds the
 *                    per-slice partials, one arrival counter per (request, KV head) and the grid barrier;
 *                    every call leaves them ready for the next call, so the zero fill is needed once.  Calls
 *                    that share a workspace must not overlap on the GPU.
 *   out            : device BF16 [total_q_rows][num_q_heads][head_dim]
 * A query row that sees no key gets zeros.  req_to_slot, seq_lens and q_row_offsets must be 4-byte
 * aligned (FTKV_ERR_ALIGN).
 * --------------------------------------------------------------------------------------------- */
size_t ftkv_decode_workspace_bytes(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t batch, int64_t total_q_rows, int32_t num_splits);

/* Number of key slices the automatic choice uses for this shape (what num_splits = 0 resolves to):
 * with few (request, KV head group) pairs, one CTA per SM; with many, enough for about eight waves of
 * resident CTAs (two per SM single-row, one when max_q_rows > 1), so that long requests are cut into
 * balanced pieces; at least ~8 keys per slice (~128 when max_q_rows > 1), at most FTKV_MAX_SPLITS. */
int32_t ftkv_decode_auto_splits(int32_t batch, int32_t num_kv_heads, int64_t max_seq_len,
                                int32_t max_q_rows);

int ftkv_decode_attn(const ftkv_pool* pool, int32_t num_q_heads, const uint16_t* q,
                     const int32_t* req_to_slot, int64_t req_stride, const int32_t* seq_lens,
                     const int32_t* q_row_offsets, int32_t batch, int64_t total_q_rows,
                     int32_t max_q_rows, int64_t max_seq_len, float sm_scale, int64_t window,
                     int32_t num_splits, uint32_t flags, void* workspace, size_t workspace_bytes,
                     uint16_t* out, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Quantize-on-write of the new tokens fused into decode: what ftkv_store_quant followed by
 * ftkv_decode_attn computes, in one launch.  The pages quantize each new K/V row when it is written
 * ([#853 "What changes"]) and then attend over the stored rows ([#897 "Fresh R9700 stage-1 A/B"]);
 * here the decode CTA whose key slice holds a new token writes that token's rows first, so a decode
 * step needs no separate store launch.
 *   k_new, v_new : device BF16 [total_q_rows][num_kv_heads][head_dim], 16-byte aligned: the K and V
 *                  rows of the new tokens, one per query row.  Query row r of request b (R rows) is
 *                  the token at position seq_lens[b] - R + r; its rows are quantized exactly as
 *                  ftkv_store_quant does and written to pool row req_to_slot[b * req_stride + that
 *                  position] before any key is read.  A position below 0 is not stored; a slot outside
 *                  the pool is flagged (ftkv_device_errors) and not written.
 * Every other argument, layout, the workspace rules, the flags and the errors are those of
 * ftkv_decode_attn; k_new or v_new NULL with work to do -> FTKV_ERR_INVALID, misaligned -> FTKV_ERR_ALIGN.
 * --------------------------------------------------------------------------------------------- */
int ftkv_decode_attn_store(const ftkv_pool* pool, int32_t num_q_heads, const uint16_t* q,
                           const uint16_t* k_new, const uint16_t* v_new, const int32_t* req_to_slot,
                           int64_t req_stride, const int32_t* seq_lens, const int32_t* q_row_offsets,
                           int32_t batch, int64_t total_q_rows, int32_t max_q_rows, int64_t max_seq_len,
                           float sm_scale, int64_t window, int32_t num_splits, uint32_t flags,
                           void* workspace, size_t workspace_bytes, uint16_t* out, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Decode without any device allocation.  The pages describe no such entry point; it exists for
 * callers that cannot allocate device memory when they need decode attention (a runtime that forbids
 * out-of-band device allocations, a plug-in that only receives buffers from its host, code that must
 * never touch an allocator).  Same arguments and results as ftkv_decode_attn, minus the workspace, the
 * flags (always 0) and the window (always 0: full attention): the split partials and arrival counters
 * live in a file-scope device array of FTKV_NOALLOC_SCRATCH_BYTES (16 MiB) that every GPU which loads
 * this library keeps until the process exits.
 *   - Every argument is checked before anything is enqueued; a refused call leaves the array untouched.
 *   - A call whose partials would not fit (roughly total_q_rows * num_q_heads * splits > 30,000 slices)
 *     returns FTKV_ERR_WORKSPACE without launching anything.
 *   - The first call on a device (with that device current) looks up the array's device address; make
 *     that first call before any stream capture.
 *   - Every call shares the array, which keeps the previous call's contents; each call clears the
 *     counters it uses on `stream`.  Calls that overlap on the GPU (other streams, other threads) race
 *     on the array: serialize them.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 * --------------------------------------------------------------------------------------------- */
#define FTKV_NOALLOC_SCRATCH_BYTES (16u << 20)

int ftkv_decode_attn_noalloc(const ftkv_pool* pool, int32_t num_q_heads, const uint16_t* q,
                             const int32_t* req_to_slot, int64_t req_stride, const int32_t* seq_lens,
                             const int32_t* q_row_offsets, int32_t batch, int64_t total_q_rows,
                             int32_t max_q_rows, int64_t max_seq_len, float sm_scale, int32_t num_splits,
                             uint16_t* out, void* stream);

/* ---------------------------------------------------------------------------------------------
 * The BF16 comparison point: the same decode and the prefill's prefix read over an unquantized BF16
 * pool, FreeToken's default KV format ("KV_FMT none" among the kernel variants of [#897] opening
 * description; FP8 is opt-in, [#853 "What changes"]).  The pages weigh FP8 against it by bytes per
 * token ([#853 "Validation"]: 98,304 BF16 vs 50,688 FP8) and by speed; these entry points let the two
 * formats run side by side on one GPU.
 *   k, v : device BF16 [num_rows][num_kv_heads][head_dim] K and V rows, caller-owned, 16-byte aligned
 * --------------------------------------------------------------------------------------------- */
typedef struct ftkv_bf16_pool {
  uint16_t* k;
  uint16_t* v;
  int64_t num_rows;
  int32_t num_kv_heads;
  int32_t head_dim;
} ftkv_bf16_pool;

/* Decode attention over a BF16 pool: for every query row, per query head i (KV head i / G),
 * o = sum_j softmax(q . k_j * sm_scale)_j v_j over the row's visible keys -- the values ftkv_decode_attn
 * computes from dequantized rows, here from the BF16 rows themselves.  Every argument, layout, flag, the
 * window, the split geometry, the workspace (ftkv_decode_workspace_bytes) and the errors are those of
 * ftkv_decode_attn, with these differences:
 *   k_new, v_new : both NULL (the new tokens' rows are already in the pool), or device BF16
 *                  [total_q_rows][num_kv_heads][head_dim]: query row r of request b (R rows) is the token at
 *                  position seq_lens[b] - R + r; its K/V rows are copied (bit for bit) to pool row
 *                  req_to_slot[b * req_stride + position], and the attention reads the new tokens from k_new /
 *                  v_new.  One NULL and the other not -> FTKV_ERR_INVALID.
 *   Every query row runs as its own set of CTAs (multi-row requests re-read their keys per row);
 *   total_q_rows above 65,535 -> FTKV_ERR_UNSUPPORTED.  FTKV_DECODE_STABLE_HISTORY takes effect only with
 *   q_row_offsets NULL.
 * --------------------------------------------------------------------------------------------- */
int ftkv_decode_attn_bf16(const ftkv_bf16_pool* pool, int32_t num_q_heads, const uint16_t* q,
                          const uint16_t* k_new, const uint16_t* v_new, const int32_t* req_to_slot,
                          int64_t req_stride, const int32_t* seq_lens, const int32_t* q_row_offsets,
                          int32_t batch, int64_t total_q_rows, int32_t max_q_rows, int64_t max_seq_len,
                          float sm_scale, int64_t window, int32_t num_splits, uint32_t flags,
                          void* workspace, size_t workspace_bytes, uint16_t* out, void* stream);

/* Prefix gather from a BF16 pool into the shared BF16 workspace, in logical order: the BF16 pool's
 * counterpart of ftkv_reconstruct_bf16, ahead of ftkv_prefill_attn / ftkv_prefill_attn_ws.
 *   slots      : device int32 [num_prefix] (4-byte aligned); logical token i lives in pool row slots[i]
 *   ws_k, ws_v : device BF16 [num_prefix][num_kv_heads][head_dim]; ws[i][h][:] = pool[slots[i]][h][:]
 * A slot outside the pool is flagged (FTKV_DEVERR_BAD_SLOT) and its workspace rows are written as zeros.
 * num_prefix == 0 is a no-op.
 * --------------------------------------------------------------------------------------------- */
int ftkv_gather_bf16(const ftkv_bf16_pool* pool, const int32_t* slots, int64_t num_prefix,
                     uint16_t* ws_k, uint16_t* ws_v, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Prefill (extend) attention of the current chunk over the reconstructed BF16 prefix plus the BF16
 * chunk itself ([#853 "What changes"]: current-chunk K/V remains BF16; [#853 "Paired end-to-end
 * A/B"]: the historical-prefix + new-token operator).
 *   q                : device BF16 [chunk_len][num_q_heads][head_dim]
 *   k_chunk, v_chunk : device BF16 [chunk_len][num_kv_heads][head_dim]
 *   ws_k, ws_v       : device BF16 [prefix_len][num_kv_heads][head_dim] (may be NULL if prefix_len 0)
 *   out              : device BF16 [chunk_len][num_q_heads][head_dim]
 * Chunk query t attends to all prefix_len prefix keys and to chunk keys 0..t.  Runs on the tcgen05
 * tensor cores (BF16 operands, FP32 accumulation in tensor memory).
 * --------------------------------------------------------------------------------------------- */
int ftkv_prefill_attn(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                      const uint16_t* q, const uint16_t* k_chunk, const uint16_t* v_chunk,
                      int64_t chunk_len, const uint16_t* ws_k, const uint16_t* ws_v,
                      int64_t prefix_len, float sm_scale, uint16_t* out, void* stream);

/* Same operation with stream-K scheduling over a caller-provided workspace (the faster entry point
 * for large chunks).  With even GQA groups the kernel takes two query heads per CTA; the work items
 * (head pair, 128-query tile) hold T = ceil(prefix_len/128) + tile + 1 key tiles.  When there are more
 * items than CTAs and each CTA's share holds a whole largest item, max_ctas persistent CTAs (<= 0: the
 * SM count) take equal ranges of all items' key tiles laid end to end; an item cut by a range boundary
 * is finished by whichever of its two pieces arrives second (partials of both in the workspace).
 * Otherwise the launch is the same as ftkv_prefill_attn.
 *   workspace       : device memory, 16-byte aligned, at least ftkv_prefill_workspace_bytes(max_ctas)
 *                     bytes, ZERO-FILLED before its first use; every call leaves its tickets at zero
 *                     again.  Calls that share a workspace must be ordered (one stream).  After a call
 *                     that raised FTKV_DEVERR_TIMEOUT the tickets may be left set: zero-fill the
 *                     workspace again before reusing it.
 * Errors: as ftkv_prefill_attn; NULL workspace -> FTKV_ERR_INVALID; too small -> FTKV_ERR_WORKSPACE;
 * unaligned -> FTKV_ERR_ALIGN.  The result is the same attention as ftkv_prefill_attn up to FP32
 * summation order (the two pieces of a cut item are combined in FP32). */
int ftkv_prefill_attn_ws(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                         const uint16_t* q, const uint16_t* k_chunk, const uint16_t* v_chunk,
                         int64_t chunk_len, const uint16_t* ws_k, const uint16_t* ws_v,
                         int64_t prefix_len, float sm_scale, int32_t max_ctas, void* workspace,
                         int64_t workspace_bytes, uint16_t* out, void* stream);

/* Workspace bytes for ftkv_prefill_attn_ws with up to max_ctas CTAs (<= 0: the current device's SM
 * count); -1 if the device cannot be queried. */
int64_t ftkv_prefill_workspace_bytes(int32_t max_ctas);

/* ---------------------------------------------------------------------------------------------
 * E4M3FN codec on the GPU, the same device code the store and attention kernels use.
 *   ftkv_e4m3_encode_f32: x device float [n] -> codes device uint8 [n]  (RNE, saturating, NaN 0x7F)
 *   ftkv_e4m3_decode_f32: codes device uint8 [n] -> x device float [n]  (exact)
 * No alignment requirement.  ([#897 "Regression and CUDA isolation"]: every finite E4M3FN value,
 * signed zero included, must survive bit-for-bit.)
 * --------------------------------------------------------------------------------------------- */
int ftkv_e4m3_encode_f32(const float* x, uint8_t* codes, int64_t n, void* stream);
int ftkv_e4m3_decode_f32(const uint8_t* codes, float* x, int64_t n, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Byte accounting ([#853 "Validation"], [#853 "Follow-up model/workload search"]), host only.
 *   bf16_bytes      = rows * layers * num_kv_heads * head_dim * 2 B * 2 (K and V)
 *   fp8_bytes       = rows * layers * 2 * num_kv_heads * (head_dim + 4)   codes + FP32 scales
 *   workspace_bytes = rows * num_kv_heads * head_dim * 2 B * 2            one shared BF16 layer
 * Any output pointer may be NULL.
 * --------------------------------------------------------------------------------------------- */
int ftkv_pool_bytes(int64_t rows, int32_t layers, int32_t num_kv_heads, int32_t head_dim,
                    int64_t* bf16_bytes, int64_t* fp8_bytes, int64_t* workspace_bytes);

/* Read and clear the current device's error word (FTKV_DEVERR_* bits).  Synchronizes the device. */
int ftkv_device_errors(int32_t* flags);

/* Human-readable name of a status code; never NULL. */
const char* ftkv_status_str(int status);

/* Text of the last CUDA error seen by this thread inside the library ("" if none). */
const char* ftkv_last_cuda_error(void);

/* ABI version (FTKV_ABI_VERSION). */
int ftkv_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FTKV_H_ */
