// ftkv_internal.h -- argument blocks and launchers shared between the C-ABI layer (api.cu) and the
// kernel translation units.  Not part of the public interface.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/ftkv.h"

namespace ftkv {

// Per-device set-up tables of the kernels cover device indices 0 .. kMaxDecodeDevices - 1.
constexpr int kMaxDecodeDevices = 64;

struct StoreArgs {
  const uint16_t* k;
  const uint16_t* v;
  const int32_t* slots;
  int64_t num_tokens;
  int num_kv_heads;
  int head_dim;              // 128 or 256
  uint8_t* k_codes;
  uint8_t* v_codes;
  float* k_scales;
  float* v_scales;
  int64_t num_rows;
  int* err;
};

struct ReconstructArgs {
  const uint8_t* k_codes;
  const uint8_t* v_codes;
  const float* k_scales;
  const float* v_scales;
  int64_t num_rows;
  int num_kv_heads;
  const int32_t* slots;
  int64_t num_prefix;
  uint16_t* ws_k;
  uint16_t* ws_v;
  int* err;
};

struct DecodeArgs {
  const uint8_t* k_codes;
  const uint8_t* v_codes;
  const float* k_scales;
  const float* v_scales;
  int64_t num_rows;
  int num_q_heads;
  int num_kv_heads;
  int group;                 // num_q_heads / num_kv_heads (1, 2, 4 or 8)
  int head_dim;              // D: 128, or 256 (single-row kernel only)
  const uint16_t* q;         // [total_q_rows][Hq][D]
  const int32_t* req_to_slot;
  int64_t req_stride;
  const int32_t* seq_lens;
  const int32_t* q_row_offsets;  // may be null: one row per request
  int batch;
  int64_t total_q_rows;
  int max_q_rows;
  int64_t max_seq_len;       // host bound used for the split geometry
  int num_splits;            // key slices per request
  int pps;                   // partials per key slice (set by the launcher); partial p of slice s of a
                             // (row, query head) is at index s * pps + p of num_splits * pps
  int64_t chunk;             // keys per slice (multiple of 16)
  float qk_scale_log2;       // sm_scale * log2(e)
  int64_t window;            // 0: full attention; W > 0: each query row attends to its last W visible keys
  int ptrans;                // partial accumulators transposed: [total_q_rows][Hq][D / 4 quads][num_splits * pps]
                             // float4 (the merge's loads of one quad over the slices are contiguous); else
                             // [total_q_rows][Hq][num_splits * pps][D] floats
  float* part_acc;
  float* part_ml;            // [total_q_rows][Hq][num_splits * pps][2]  (max in log2 units, sum)
  int* counters;             // [batch][Hkv] arrival tickets; zero between calls
  uint16_t* out;             // [total_q_rows][Hq][D]
  int* err;
  int early;                 // FTKV_DECODE_STABLE_HISTORY: history loads may start before the preceding grid ends
  int scan_scales;           // the slot tables may cover most of the pool: bring the scale arrays into L2 whole
  int coop;                  // set by the launcher: cooperative launch, merge after a grid barrier
  int* gbar;                 // [2] grid barrier: arrivals of every call so far, and their count when the
                             // previous call's barrier completed (zero-filled once; no reset between calls)
  const uint16_t* k_new;     // fused store: [total_q_rows][Hkv][128] K of the new tokens, or null
  const uint16_t* v_new;     //              V of the new tokens
  const uint16_t* k_bf16;    // BF16 pool (decode_bf16 only): [num_rows][Hkv][128] K rows
  const uint16_t* v_bf16;    //                               V rows
};

// Prefix gather from a BF16 pool into the shared workspace (the BF16 counterpart of reconstruction).
struct GatherArgs {
  const uint16_t* k;         // [num_rows][Hkv][128]
  const uint16_t* v;
  int64_t num_rows;
  int num_kv_heads;
  const int32_t* slots;      // [num_prefix]
  int64_t num_prefix;
  uint16_t* ws_k;            // [num_prefix][Hkv][128]
  uint16_t* ws_v;
  int* err;
};

struct PrefillArgs {
  int num_q_heads;
  int num_kv_heads;
  const uint16_t* q;         // [C][Hq][128]
  const uint16_t* k_chunk;   // [C][Hkv][128]
  const uint16_t* v_chunk;
  int64_t chunk_len;
  const uint16_t* ws_k;      // [P][Hkv][128]
  const uint16_t* ws_v;
  int64_t prefix_len;
  float qk_scale_log2;
  uint16_t* out;             // [C][Hq][128]
  int* err;
  // stream-K scheduling of the two-heads-per-CTA kernel (tcgen05 path): workspace, or null for one CTA
  // per work item; max_ctas <= 0 means the SM count
  void* workspace;
  int64_t workspace_bytes;
  int max_ctas;
};

// Bytes of the stream-K prefill workspace for up to max_ctas persistent CTAs (see launch_prefill_tc).
int64_t prefill_workspace_bytes(int max_ctas);

// Launch with programmatic stream serialization (see pdl_enter in ftkv_device.cuh).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Same, as a cooperative launch: every CTA of the grid is resident at once (the launch fails otherwise).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k_coop(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                 Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2]{};
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

cudaError_t launch_store_quant(const StoreArgs& a, cudaStream_t s);
cudaError_t launch_reconstruct(const ReconstructArgs& a, cudaStream_t s);
cudaError_t launch_e4m3_encode(const float* x, uint8_t* c, int64_t n, int num_sms, cudaStream_t s);
cudaError_t launch_e4m3_decode(const uint8_t* c, float* x, int64_t n, int num_sms, cudaStream_t s);
// Decode (decode.cu): single-row batches run the token-major kernel (decode_tok.cu), multi-row batches the
// tensor-memory kernel with one KV head per CTA (decode_mr.cu: max_q_rows > 1, 128-d heads).
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_mr(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_tok(const DecodeArgs& a, cudaStream_t s);
// Decode over a BF16 pool (bf16_pool.cu): one grid row per query row, any number of rows per request.
cudaError_t launch_decode_bf16(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_gather_bf16(const GatherArgs& a, cudaStream_t s);
int decode_ctas_per_sm(int max_q_rows);
int decode_tok_heads_per_cta(int num_kv_heads);
cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s);

// Host-side checks and split geometry of a decode call, shared by every decode entry point.  Returns
// FTKV_OK or the status the entry point reports; nothing is enqueued.  `workspace` is not checked when
// check_workspace is false (the allocation-free entry point supplies its own).
struct DecodeGeom {
  int64_t splits = 0;   // key slices per request
  int64_t parts = 0;    // partial slots in the workspace (rows x query heads x slices x partials per slice)
  int64_t chunk = 0;    // keys per slice
  int64_t span = 0;     // most keys one request attends to (max_seq_len, or less with a sliding window)
  size_t need = 0;      // workspace bytes
  bool empty = false;   // nothing to compute (batch or total_q_rows is 0)
};
// Every argument check of a decode call except the pool's (the caller checks its pool first), and the split
// geometry.
int decode_validate_dims(int32_t num_kv_heads, int32_t head_dim, int32_t num_q_heads, const uint16_t* q,
                         const int32_t* req_to_slot, int64_t req_stride, const int32_t* seq_lens, const int32_t* q_row_offsets, int32_t batch,
                         int64_t total_q_rows, int32_t max_q_rows, int64_t max_seq_len, float sm_scale,
                         int64_t window, int32_t num_splits, uint32_t flags, const void* workspace,
                         size_t workspace_bytes, const uint16_t* out, bool check_workspace, DecodeGeom* geom);
// The FP8 pool's checks, then decode_validate_dims.
int decode_validate(const ftkv_pool* pool, int32_t num_q_heads, const uint16_t* q, const int32_t* req_to_slot,
                    int64_t req_stride, const int32_t* seq_lens, const int32_t* q_row_offsets, int32_t batch,
                    int64_t total_q_rows, int32_t max_q_rows, int64_t max_seq_len, float sm_scale,
                    int64_t window, int32_t num_splits, uint32_t flags, const void* workspace,
                    size_t workspace_bytes, const uint16_t* out, bool check_workspace, DecodeGeom* geom);

}  // namespace ftkv
