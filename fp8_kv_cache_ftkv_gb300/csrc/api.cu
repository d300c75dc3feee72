// api.cu -- the extern "C" entry points of libftkv.so (declared in include/ftkv.h).
//
// Every entry point validates its arguments on the host and returns a status before anything is
// enqueued; kernels are launched on the caller's stream and never allocate.  The per-device error
// word (slots outside the pool, sequence lengths above the declared bound) is a 4-byte __device__
// variable of this translation unit whose address is handed to the kernels.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/ftkv.h"
#include "ftkv_internal.h"

namespace {

__device__ int g_device_errors;

thread_local char g_last_cuda_error[256] = "";

int cuda_fail(cudaError_t e) {
  std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", cudaGetErrorName(e),
                cudaGetErrorString(e));
  return FTKV_ERR_CUDA;
}

struct DeviceInfo {
  int num_sms = 0;
  int* err_word = nullptr;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
std::mutex g_info_mu;

// Per-device set-up: SM count and the device address of the error word.
int device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return FTKV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_info_mu);
  DeviceInfo& di = g_info[dev];
  if (di.num_sms == 0) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_errors);
    if (e != cudaSuccess) return cuda_fail(e);
    di.err_word = static_cast<int*>(p);
    di.num_sms = sms;
  }
  *out = &di;
  return FTKV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_pool(const ftkv_pool* pool) {
  if (!pool || !pool->k_codes || !pool->v_codes || !pool->k_scales || !pool->v_scales) return FTKV_ERR_INVALID;
  if (pool->num_rows <= 0 || pool->num_kv_heads <= 0 || pool->num_rows > (int64_t(1) << 31) - 1)
    return FTKV_ERR_INVALID;
  if (pool->head_dim != FTKV_HEAD_DIM && pool->head_dim != FTKV_HEAD_DIM_256) return FTKV_ERR_UNSUPPORTED;
  if (!aligned16(pool->k_codes) || !aligned16(pool->v_codes)) return FTKV_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(pool->k_scales) & 3u) || (reinterpret_cast<uintptr_t>(pool->v_scales) & 3u))
    return FTKV_ERR_ALIGN;
  return FTKV_OK;
}

int check_bf16_pool(const ftkv_bf16_pool* pool) {
  if (!pool || !pool->k || !pool->v) return FTKV_ERR_INVALID;
  if (pool->num_rows <= 0 || pool->num_kv_heads <= 0 || pool->num_rows > (int64_t(1) << 31) - 1)
    return FTKV_ERR_INVALID;
  if (pool->head_dim != FTKV_HEAD_DIM) return FTKV_ERR_UNSUPPORTED;
  if (!aligned16(pool->k) || !aligned16(pool->v)) return FTKV_ERR_ALIGN;
  return FTKV_OK;
}

int check_heads(int32_t hq, int32_t hkv) {
  if (hq <= 0 || hkv <= 0) return FTKV_ERR_INVALID;
  if (hq % hkv != 0) return FTKV_ERR_UNSUPPORTED;
  const int g = hq / hkv;
  if (g != 1 && g != 2 && g != 4 && g != 8) return FTKV_ERR_UNSUPPORTED;
  return FTKV_OK;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

extern "C" {

int ftkv_abi_version(void) { return FTKV_ABI_VERSION; }

const char* ftkv_status_str(int status) {
  switch (status) {
    case FTKV_OK: return "FTKV_OK";
    case FTKV_ERR_INVALID: return "FTKV_ERR_INVALID";
    case FTKV_ERR_UNSUPPORTED: return "FTKV_ERR_UNSUPPORTED";
    case FTKV_ERR_ALIGN: return "FTKV_ERR_ALIGN";
    case FTKV_ERR_WORKSPACE: return "FTKV_ERR_WORKSPACE";
    case FTKV_ERR_CUDA: return "FTKV_ERR_CUDA";
    default: return "FTKV_ERR_UNKNOWN";
  }
}

const char* ftkv_last_cuda_error(void) { return g_last_cuda_error; }

int ftkv_pool_bytes(int64_t rows, int32_t layers, int32_t num_kv_heads, int32_t head_dim,
                    int64_t* bf16_bytes, int64_t* fp8_bytes, int64_t* workspace_bytes) {
  if (rows < 0 || layers < 0 || num_kv_heads <= 0 || head_dim <= 0) return FTKV_ERR_INVALID;
  const int64_t per_row_bf16 = int64_t(num_kv_heads) * head_dim * 2 * 2;
  const int64_t per_row_fp8 = 2 * int64_t(num_kv_heads) * (head_dim + 4);
  if (bf16_bytes) *bf16_bytes = rows * layers * per_row_bf16;
  if (fp8_bytes) *fp8_bytes = rows * layers * per_row_fp8;
  if (workspace_bytes) *workspace_bytes = rows * per_row_bf16;
  return FTKV_OK;
}

int ftkv_store_quant(const ftkv_pool* pool, const uint16_t* k, const uint16_t* v, const int32_t* slots,
                     int64_t num_tokens, void* stream) {
  int st = check_pool(pool);
  if (st != FTKV_OK) return st;
  if (num_tokens < 0) return FTKV_ERR_INVALID;
  if (num_tokens == 0) return FTKV_OK;
  if (!k || !v || !slots) return FTKV_ERR_INVALID;
  if (!aligned16(k) || !aligned16(v) || (reinterpret_cast<uintptr_t>(slots) & 3u)) return FTKV_ERR_ALIGN;
  DeviceInfo* di = nullptr;
  if ((st = device_info(&di)) != FTKV_OK) return st;
  ftkv::StoreArgs a{k, v, slots, num_tokens, pool->num_kv_heads, pool->head_dim, pool->k_codes, pool->v_codes,
                    pool->k_scales, pool->v_scales, pool->num_rows, di->err_word};
  cudaError_t e = ftkv::launch_store_quant(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FTKV_OK : cuda_fail(e);
}

int ftkv_reconstruct_bf16(const ftkv_pool* pool, const int32_t* slots, int64_t num_prefix, uint16_t* ws_k,
                          uint16_t* ws_v, void* stream) {
  int st = check_pool(pool);
  if (st != FTKV_OK) return st;
  if (pool->head_dim != FTKV_HEAD_DIM) return FTKV_ERR_UNSUPPORTED;  // the prefill path is 128-d
  if (num_prefix < 0) return FTKV_ERR_INVALID;
  if (num_prefix == 0) return FTKV_OK;
  if (!slots || !ws_k || !ws_v) return FTKV_ERR_INVALID;
  if (!aligned16(ws_k) || !aligned16(ws_v) || (reinterpret_cast<uintptr_t>(slots) & 3u)) return FTKV_ERR_ALIGN;
  DeviceInfo* di = nullptr;
  if ((st = device_info(&di)) != FTKV_OK) return st;
  ftkv::ReconstructArgs a{pool->k_codes, pool->v_codes, pool->k_scales, pool->v_scales, pool->num_rows,
                          pool->num_kv_heads, slots, num_prefix, ws_k, ws_v, di->err_word};
  cudaError_t e = ftkv::launch_reconstruct(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FTKV_OK : cuda_fail(e);
}

// Workspace layout: [partial accumulators | partial (max, sum) | arrival counters], 256-B aligned parts.
static int64_t ws_acc_bytes(int64_t parts, int head_dim) { return ceil_div(parts * head_dim * 4, 256) * 256; }
static int64_t ws_ml_bytes(int64_t parts) { return ceil_div(parts * 2 * 4, 256) * 256; }

size_t ftkv_decode_workspace_bytes(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t batch,
                                   int64_t total_q_rows, int32_t num_splits) {
  if (num_q_heads <= 0 || num_kv_heads <= 0 || batch < 0 || total_q_rows < 0 ||
      (head_dim != FTKV_HEAD_DIM && head_dim != FTKV_HEAD_DIM_256))
    return 0;
  if (num_splits <= 0 || num_splits > FTKV_MAX_SPLITS) num_splits = FTKV_MAX_SPLITS;
  const int64_t parts = total_q_rows * num_q_heads * num_splits;  // one partial per (row, query head, slice)
  const int64_t ctr = ceil_div((int64_t(batch) * num_kv_heads + 2) * 4, 256) * 256;  // + the grid barrier
  return static_cast<size_t>(ws_acc_bytes(parts, head_dim) + ws_ml_bytes(parts) + ctr);
}

int32_t ftkv_decode_auto_splits(int32_t batch, int32_t num_kv_heads, int64_t max_seq_len, int32_t max_q_rows) {
  if (batch <= 0 || num_kv_heads <= 0 || max_seq_len <= 0) return 1;
  DeviceInfo* di = nullptr;
  int sms = 152;
  if (device_info(&di) == FTKV_OK) sms = di->num_sms;
  const int64_t per_sm = ftkv::decode_ctas_per_sm(max_q_rows);
  // A CTA of the single-row kernel covers every KV head of its keys (up to 4 per CTA); the multi-row kernel
  // takes one KV head per CTA.
  const int64_t heads_per_cta = max_q_rows <= 1 ? ftkv::decode_tok_heads_per_cta(num_kv_heads) : 1;
  const int64_t groups = int64_t(batch) * (num_kv_heads / heads_per_cta);
  // Single-row kernel (two CTAs fit per SM):
  //  * at most 4 (request, head group) pairs: one CTA per SM.  The grid is resident at once and merges
  //    cooperatively, and the other CTA slot of every SM is left to the next launch in the stream (batch 1,
  //    32K keys, 48 layers: 152 slices 675 us per step, 76-200 slices 940-1,140 us);
  //  * more: whole waves of resident CTAs (two per SM), as few as give at least ~8 slices (8-layer chains of
  //    16,384-key requests, per layer: 16 requests 114 us at one CTA per SM, 67 us at one wave of two;
  //    32 requests 165 us at ~8 waves, 129 us at one or two; 64 requests 274 us at 1.7 waves, 253 us at 4;
  //    4 requests 25.5 us either way).
  // Multi-row kernel (one CTA per SM): few pairs (at most one per 8 SMs) one CTA per SM; many, about 8 waves
  // (64 requests of 1-8 rows, 4 KV heads: 4 slices 746 us, 5 slices 748 us, 8 slices 758 us, 10 slices
  // 779 us: every multi-row CTA pays its pipeline's fill and drain).
  int64_t s;
  if (max_q_rows <= 1)
    s = (groups <= 4) ? sms / groups
                      : std::max<int64_t>(1, ceil_div(8 * groups, per_sm * sms)) * per_sm * sms / groups;
  else
    s = (8 * groups <= sms) ? sms / groups : ceil_div(8 * sms * per_sm, groups);
  // at least ~8 keys per slice for the single-row kernel: short requests still spread over the SMs, and the
  // split merge with them (512 keys, batch 1, one call: 16 slices 20.5 us, 32 slices 14.4 us, 64 or more
  // 12.3 us); ~128 (one tile) for the multi-row kernel
  const int64_t by_len = ceil_div(max_seq_len, max_q_rows <= 1 ? 8 : 128);
  if (s > by_len) s = by_len;
  if (s > FTKV_MAX_SPLITS) s = FTKV_MAX_SPLITS;
  if (s < 1) s = 1;
  return static_cast<int32_t>(s);
}

}  // extern "C"

namespace ftkv {

int decode_validate_dims(int32_t num_kv_heads, int32_t head_dim, int32_t num_q_heads, const uint16_t* q, const int32_t* req_to_slot,
                         int64_t req_stride, const int32_t* seq_lens, const int32_t* q_row_offsets, int32_t batch,
                         int64_t total_q_rows, int32_t max_q_rows, int64_t max_seq_len, float sm_scale,
                         int64_t window, int32_t num_splits, uint32_t flags, const void* workspace,
                         size_t workspace_bytes, const uint16_t* out, bool check_workspace, DecodeGeom* geom) {
  *geom = DecodeGeom{};
  int st;
  if ((st = check_heads(num_q_heads, num_kv_heads)) != FTKV_OK) return st;
  if (head_dim != FTKV_HEAD_DIM && head_dim != FTKV_HEAD_DIM_256) return FTKV_ERR_UNSUPPORTED;
  if (batch < 0 || total_q_rows < 0 || max_seq_len < 0 || req_stride < 0) return FTKV_ERR_INVALID;
  if (max_q_rows < 1 || max_q_rows > FTKV_MAX_Q_ROWS) return FTKV_ERR_UNSUPPORTED;
  if (batch > FTKV_MAX_BATCH) return FTKV_ERR_UNSUPPORTED;  // the requests are one grid dimension
  if (head_dim == FTKV_HEAD_DIM_256 && max_q_rows > 1) return FTKV_ERR_UNSUPPORTED;  // single-row kernel only
  if (num_splits < 0 || num_splits > FTKV_MAX_SPLITS) return FTKV_ERR_INVALID;
  if (flags & ~static_cast<uint32_t>(FTKV_DECODE_STABLE_HISTORY)) return FTKV_ERR_INVALID;
  if (max_seq_len > req_stride) return FTKV_ERR_INVALID;
  if (max_seq_len > (int64_t(1) << 31) - 1 - 4096) return FTKV_ERR_UNSUPPORTED;
  if (!q_row_offsets && total_q_rows != batch) return FTKV_ERR_INVALID;
  if (total_q_rows > int64_t(batch) * max_q_rows) return FTKV_ERR_INVALID;
  if (!(sm_scale == sm_scale)) return FTKV_ERR_INVALID;
  if (window < 0) return FTKV_ERR_INVALID;
  if (batch == 0 || total_q_rows == 0) {
    geom->empty = true;
    return FTKV_OK;
  }
  if (!q || !req_to_slot || !seq_lens || !out || (check_workspace && !workspace)) return FTKV_ERR_INVALID;
  if (!aligned16(q) || !aligned16(out)) return FTKV_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(req_to_slot) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(q_row_offsets) & 3u))
    return FTKV_ERR_ALIGN;
  if (check_workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return FTKV_ERR_ALIGN;
  if (total_q_rows > (int64_t(1) << 31) - 1) return FTKV_ERR_UNSUPPORTED;

  // Keys a request attends to at most: all of them, or with a sliding window of W keys the last W + R - 1
  // (the union of its R rows' windows); the slices cover only those.
  const int64_t span = (window > 0 && window + max_q_rows - 1 < max_seq_len) ? window + max_q_rows - 1 : max_seq_len;
  geom->span = span;
  if (num_splits == 0) num_splits = ftkv_decode_auto_splits(batch, num_kv_heads, span, max_q_rows);
  // keys per slice: a multiple of 8 for the single-row kernel (its blocks of 16 keys may end inside a slice),
  // of 16 for the multi-row kernel
  const int64_t align = max_q_rows <= 1 ? 8 : 16;
  int64_t chunk = ceil_div(span > 0 ? span : 1, num_splits);
  chunk = ceil_div(chunk, align) * align;
  geom->chunk = chunk;
  geom->splits = span > 0 ? ceil_div(span, chunk) : 1;
  geom->need = ftkv_decode_workspace_bytes(num_q_heads, num_kv_heads, head_dim, batch, total_q_rows,
                                           static_cast<int32_t>(geom->splits));
  geom->parts = total_q_rows * num_q_heads * geom->splits;
  if (check_workspace && workspace_bytes < geom->need) return FTKV_ERR_WORKSPACE;
  return FTKV_OK;
}

int decode_validate(const ftkv_pool* pool, int32_t num_q_heads, const uint16_t* q, const int32_t* req_to_slot,
                    int64_t req_stride, const int32_t* seq_lens, const int32_t* q_row_offsets, int32_t batch,
                    int64_t total_q_rows, int32_t max_q_rows, int64_t max_seq_len, float sm_scale,
                    int64_t window, int32_t num_splits, uint32_t flags, const void* workspace,
                    size_t workspace_bytes, const uint16_t* out, bool check_workspace, DecodeGeom* geom) {
  *geom = DecodeGeom{};
  const int st = check_pool(pool);
  if (st != FTKV_OK) return st;
  return decode_validate_dims(pool->num_kv_heads, pool->head_dim, num_q_heads, q, req_to_slot, req_stride, seq_lens, q_row_offsets,
                              batch, total_q_rows, max_q_rows, max_seq_len, sm_scale, window, num_splits, flags,
                              workspace, workspace_bytes, out, check_workspace, geom);
}

}  // namespace ftkv

extern "C" {

static int decode_common(const ftkv_pool* pool, int32_t num_q_heads, const uint16_t* q, const int32_t* req_to_slot,
                         int64_t req_stride, const int32_t* seq_lens, const int32_t* q_row_offsets, int32_t batch,
                         int64_t total_q_rows, int32_t max_q_rows, int64_t max_seq_len, float sm_scale,
                         int64_t window, int32_t num_splits, uint32_t flags, void* workspace,
                         size_t workspace_bytes, uint16_t* out, void* stream, const uint16_t* k_new = nullptr,
                         const uint16_t* v_new = nullptr) {
  ftkv::DecodeGeom geom;
  int st = ftkv::decode_validate(pool, num_q_heads, q, req_to_slot, req_stride, seq_lens, q_row_offsets, batch,
                                 total_q_rows, max_q_rows, max_seq_len, sm_scale, window, num_splits, flags,
                                 workspace, workspace_bytes, out, true, &geom);
  if (st != FTKV_OK || geom.empty) return st;
  DeviceInfo* di = nullptr;
  if ((st = device_info(&di)) != FTKV_OK) return st;
  const int64_t parts = geom.parts;  // the layout ftkv_decode_workspace_bytes sizes
  float* part_acc = static_cast<float*>(workspace);
  char* ws = static_cast<char*>(workspace);
  float* part_ml = reinterpret_cast<float*>(ws + ws_acc_bytes(parts, pool->head_dim));
  int* counters = reinterpret_cast<int*>(ws + ws_acc_bytes(parts, pool->head_dim) + ws_ml_bytes(parts));

  ftkv::DecodeArgs a{};
  a.k_codes = pool->k_codes;
  a.v_codes = pool->v_codes;
  a.k_scales = pool->k_scales;
  a.v_scales = pool->v_scales;
  a.num_rows = pool->num_rows;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = pool->num_kv_heads;
  a.group = num_q_heads / pool->num_kv_heads;
  a.head_dim = pool->head_dim;
  a.q = q;
  a.req_to_slot = req_to_slot;
  a.req_stride = req_stride;
  a.seq_lens = seq_lens;
  a.q_row_offsets = q_row_offsets;
  a.batch = batch;
  a.total_q_rows = total_q_rows;
  a.max_q_rows = max_q_rows;
  a.max_seq_len = max_seq_len;
  a.num_splits = static_cast<int>(geom.splits);
  a.chunk = geom.chunk;
  a.qk_scale_log2 = sm_scale * 1.4426950408889634f;
  a.window = window;
  a.part_acc = part_acc;
  a.part_ml = part_ml;
  a.counters = counters;
  a.gbar = counters + int64_t(batch) * pool->num_kv_heads;
  a.out = out;
  a.err = di->err_word;
  a.early = (flags & FTKV_DECODE_STABLE_HISTORY) ? 1 : 0;
  // When the requests' keys may cover at least half of the pool rows, the kernel reads the scale arrays
  // into L2 sequentially at its start instead of leaving them to scattered 4-byte reads.
  a.scan_scales = (int64_t(batch) * geom.span * 2 >= pool->num_rows) ? 1 : 0;
  a.k_new = k_new;
  a.v_new = v_new;
  cudaError_t e = ftkv::launch_decode(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FTKV_OK : cuda_fail(e);
}

int ftkv_decode_attn(const ftkv_pool* pool, int32_t num_q_heads, const uint16_t* q, const int32_t* req_to_slot,
                     int64_t req_stride, const int32_t* seq_lens, const int32_t* q_row_offsets, int32_t batch,
                     int64_t total_q_rows, int32_t max_q_rows, int64_t max_seq_len, float sm_scale,
                     int64_t window, int32_t num_splits, uint32_t flags, void* workspace, size_t workspace_bytes,
                     uint16_t* out, void* stream) {
  return decode_common(pool, num_q_heads, q, req_to_slot, req_stride, seq_lens, q_row_offsets, batch, total_q_rows,
                       max_q_rows, max_seq_len, sm_scale, window, num_splits, flags, workspace, workspace_bytes, out,
                       stream);
}

int ftkv_decode_attn_store(const ftkv_pool* pool, int32_t num_q_heads, const uint16_t* q, const uint16_t* k_new,
                           const uint16_t* v_new, const int32_t* req_to_slot, int64_t req_stride,
                           const int32_t* seq_lens, const int32_t* q_row_offsets, int32_t batch, int64_t total_q_rows,
                           int32_t max_q_rows, int64_t max_seq_len, float sm_scale, int64_t window,
                           int32_t num_splits, uint32_t flags, void* workspace, size_t workspace_bytes, uint16_t* out,
                           void* stream) {
  if (batch > 0 && total_q_rows > 0) {
    if (!k_new || !v_new) return FTKV_ERR_INVALID;
    if (!aligned16(k_new) || !aligned16(v_new)) return FTKV_ERR_ALIGN;
  }
  return decode_common(pool, num_q_heads, q, req_to_slot, req_stride, seq_lens, q_row_offsets, batch, total_q_rows,
                       max_q_rows, max_seq_len, sm_scale, window, num_splits, flags, workspace, workspace_bytes, out,
                       stream, k_new, v_new);
}

int ftkv_decode_attn_bf16(const ftkv_bf16_pool* pool, int32_t num_q_heads, const uint16_t* q, const uint16_t* k_new,
                          const uint16_t* v_new, const int32_t* req_to_slot, int64_t req_stride,
                          const int32_t* seq_lens, const int32_t* q_row_offsets, int32_t batch, int64_t total_q_rows,
                          int32_t max_q_rows, int64_t max_seq_len, float sm_scale, int64_t window,
                          int32_t num_splits, uint32_t flags, void* workspace, size_t workspace_bytes, uint16_t* out,
                          void* stream) {
  int st = check_bf16_pool(pool);
  if (st != FTKV_OK) return st;
  ftkv::DecodeGeom geom;
  st = ftkv::decode_validate_dims(pool->num_kv_heads, FTKV_HEAD_DIM, num_q_heads, q, req_to_slot, req_stride, seq_lens,
                                  q_row_offsets, batch, total_q_rows, max_q_rows, max_seq_len, sm_scale, window,
                                  num_splits, flags, workspace, workspace_bytes, out, true, &geom);
  if (st != FTKV_OK || geom.empty) return st;
  if ((k_new == nullptr) != (v_new == nullptr)) return FTKV_ERR_INVALID;
  if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return FTKV_ERR_ALIGN;
  if (total_q_rows > 65535) return FTKV_ERR_UNSUPPORTED;  // one grid row per query row
  DeviceInfo* di = nullptr;
  if ((st = device_info(&di)) != FTKV_OK) return st;
  char* ws = static_cast<char*>(workspace);
  ftkv::DecodeArgs a{};
  a.num_rows = pool->num_rows;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = pool->num_kv_heads;
  a.group = num_q_heads / pool->num_kv_heads;
  a.head_dim = FTKV_HEAD_DIM;
  a.q = q;
  a.req_to_slot = req_to_slot;
  a.req_stride = req_stride;
  a.seq_lens = seq_lens;
  a.q_row_offsets = q_row_offsets;
  a.batch = batch;
  a.total_q_rows = total_q_rows;
  a.max_q_rows = max_q_rows;
  a.max_seq_len = max_seq_len;
  a.num_splits = static_cast<int>(geom.splits);
  a.chunk = geom.chunk;
  a.qk_scale_log2 = sm_scale * 1.4426950408889634f;
  a.window = window;
  a.part_acc = static_cast<float*>(workspace);  // the layout ftkv_decode_workspace_bytes sizes
  a.part_ml = reinterpret_cast<float*>(ws + ws_acc_bytes(geom.parts, FTKV_HEAD_DIM));
  a.counters = reinterpret_cast<int*>(ws + ws_acc_bytes(geom.parts, FTKV_HEAD_DIM) + ws_ml_bytes(geom.parts));
  a.gbar = a.counters + int64_t(batch) * pool->num_kv_heads;
  a.out = out;
  a.err = di->err_word;
  a.early = (flags & FTKV_DECODE_STABLE_HISTORY) ? 1 : 0;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_bf16 = pool->k;
  a.v_bf16 = pool->v;
  cudaError_t e = ftkv::launch_decode_bf16(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FTKV_OK : cuda_fail(e);
}

int ftkv_gather_bf16(const ftkv_bf16_pool* pool, const int32_t* slots, int64_t num_prefix, uint16_t* ws_k,
                     uint16_t* ws_v, void* stream) {
  int st = check_bf16_pool(pool);
  if (st != FTKV_OK) return st;
  if (num_prefix < 0) return FTKV_ERR_INVALID;
  if (num_prefix == 0) return FTKV_OK;
  if (!slots || !ws_k || !ws_v) return FTKV_ERR_INVALID;
  if (!aligned16(ws_k) || !aligned16(ws_v) || (reinterpret_cast<uintptr_t>(slots) & 3u)) return FTKV_ERR_ALIGN;
  DeviceInfo* di = nullptr;
  if ((st = device_info(&di)) != FTKV_OK) return st;
  ftkv::GatherArgs a{pool->k, pool->v, pool->num_rows, pool->num_kv_heads, slots, num_prefix, ws_k, ws_v,
                     di->err_word};
  cudaError_t e = ftkv::launch_gather_bf16(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FTKV_OK : cuda_fail(e);
}

static int prefill_common(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, const uint16_t* q,
                          const uint16_t* k_chunk, const uint16_t* v_chunk, int64_t chunk_len,
                          const uint16_t* ws_k, const uint16_t* ws_v, int64_t prefix_len, float sm_scale,
                          uint16_t* out, void* stream, int32_t max_ctas = 0, void* workspace = nullptr,
                          int64_t workspace_bytes = 0) {
  int st = check_heads(num_q_heads, num_kv_heads);
  if (st != FTKV_OK) return st;
  if (head_dim != FTKV_HEAD_DIM) return FTKV_ERR_UNSUPPORTED;
  if (chunk_len < 0 || prefix_len < 0) return FTKV_ERR_INVALID;
  if (!(sm_scale == sm_scale)) return FTKV_ERR_INVALID;
  if (chunk_len == 0) return FTKV_OK;
  if (!q || !k_chunk || !v_chunk || !out) return FTKV_ERR_INVALID;
  if (prefix_len > 0 && (!ws_k || !ws_v)) return FTKV_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_chunk) || !aligned16(v_chunk) || !aligned16(out)) return FTKV_ERR_ALIGN;
  if (prefix_len > 0 && (!aligned16(ws_k) || !aligned16(ws_v))) return FTKV_ERR_ALIGN;
  if (chunk_len > (int64_t(1) << 31) - 1 || prefix_len > (int64_t(1) << 31) - 1) return FTKV_ERR_UNSUPPORTED;
  DeviceInfo* di = nullptr;
  if ((st = device_info(&di)) != FTKV_OK) return st;
  if (workspace) {
    if (!aligned16(workspace)) return FTKV_ERR_ALIGN;
    if (workspace_bytes < ftkv::prefill_workspace_bytes(max_ctas > 0 ? max_ctas : di->num_sms))
      return FTKV_ERR_WORKSPACE;
  }
  ftkv::PrefillArgs a{num_q_heads, num_kv_heads, q, k_chunk, v_chunk, chunk_len,
                      prefix_len > 0 ? ws_k : k_chunk, prefix_len > 0 ? ws_v : v_chunk, prefix_len,
                      sm_scale * 1.4426950408889634f, out, di->err_word, workspace, workspace_bytes,
                      max_ctas};
  cudaError_t e = ftkv::launch_prefill_tc(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FTKV_OK : cuda_fail(e);
}

int ftkv_prefill_attn(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, const uint16_t* q,
                      const uint16_t* k_chunk, const uint16_t* v_chunk, int64_t chunk_len, const uint16_t* ws_k,
                      const uint16_t* ws_v, int64_t prefix_len, float sm_scale, uint16_t* out, void* stream) {
  return prefill_common(num_q_heads, num_kv_heads, head_dim, q, k_chunk, v_chunk, chunk_len, ws_k, ws_v,
                        prefix_len, sm_scale, out, stream);
}

int ftkv_prefill_attn_ws(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, const uint16_t* q,
                         const uint16_t* k_chunk, const uint16_t* v_chunk, int64_t chunk_len, const uint16_t* ws_k,
                         const uint16_t* ws_v, int64_t prefix_len, float sm_scale, int32_t max_ctas,
                         void* workspace, int64_t workspace_bytes, uint16_t* out, void* stream) {
  if (!workspace || workspace_bytes < 0) return FTKV_ERR_INVALID;
  return prefill_common(num_q_heads, num_kv_heads, head_dim, q, k_chunk, v_chunk, chunk_len, ws_k, ws_v,
                        prefix_len, sm_scale, out, stream, max_ctas, workspace, workspace_bytes);
}

int64_t ftkv_prefill_workspace_bytes(int32_t max_ctas) {
  if (max_ctas <= 0) {
    DeviceInfo* di = nullptr;
    if (device_info(&di) != FTKV_OK) return -1;
    max_ctas = di->num_sms;
  }
  return ftkv::prefill_workspace_bytes(max_ctas);
}

int ftkv_e4m3_encode_f32(const float* x, uint8_t* codes, int64_t n, void* stream) {
  if (n < 0) return FTKV_ERR_INVALID;
  if (n == 0) return FTKV_OK;
  if (!x || !codes) return FTKV_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(x) & 3u) return FTKV_ERR_ALIGN;
  DeviceInfo* di = nullptr;
  int st = device_info(&di);
  if (st != FTKV_OK) return st;
  cudaError_t e = ftkv::launch_e4m3_encode(x, codes, n, di->num_sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FTKV_OK : cuda_fail(e);
}

int ftkv_e4m3_decode_f32(const uint8_t* codes, float* x, int64_t n, void* stream) {
  if (n < 0) return FTKV_ERR_INVALID;
  if (n == 0) return FTKV_OK;
  if (!x || !codes) return FTKV_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(x) & 3u) return FTKV_ERR_ALIGN;
  DeviceInfo* di = nullptr;
  int st = device_info(&di);
  if (st != FTKV_OK) return st;
  cudaError_t e = ftkv::launch_e4m3_decode(codes, x, n, di->num_sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FTKV_OK : cuda_fail(e);
}

int ftkv_device_errors(int32_t* flags) {
  if (!flags) return FTKV_ERR_INVALID;
  DeviceInfo* di = nullptr;
  int st = device_info(&di);
  if (st != FTKV_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  int v = 0;
  e = cudaMemcpy(&v, di->err_word, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  const int zero = 0;
  e = cudaMemcpy(di->err_word, &zero, sizeof(int), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e);
  *flags = v;
  return FTKV_OK;
}

}  // extern "C"
