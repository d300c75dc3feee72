// decode_noalloc.cu -- split-K decode attention for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc (or any allocator) at the point where they need
// decode attention: code that runs inside a memory-accounting runtime that forbids out-of-band device
// allocations, plugins handed a fixed set of buffers by their host, or code paths that must not touch
// the allocator at all.  ftkv_decode_attn_noalloc serves them: the caller still passes every input and
// the output, and the split partials and arrival counters live in a file-scope device array of
// FTKV_NOALLOC_SCRATCH_BYTES that every GPU loading this library holds until the process exits.
//
// Set-up: the first call on a device (with that device current) obtains the array's device address
// with cudaGetSymbolAddress and keeps it; in host code the array's name is only a host-side stand-in
// and must never be handed to a kernel.  Make that first call before any stream capture.
// Every call shares the one array and it keeps the previous call's contents, so each call clears the
// arrival counters it is about to use (cudaMemsetAsync on the caller's stream), after every argument has
// been checked: a call that is refused enqueues nothing.  Calls that overlap on the GPU -- on different
// streams, or from different threads -- race on the array; serialize them.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/ftkv.h"
#include "ftkv_internal.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[FTKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

int64_t round256(int64_t x) { return (x + 255) / 256 * 256; }

// Device address of the scratch array for the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FTKV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FTKV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FTKV_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FTKV_OK;
}

}  // namespace

extern "C" int ftkv_decode_attn_noalloc(const ftkv_pool* pool, int32_t num_q_heads, const uint16_t* q,
                                        const int32_t* req_to_slot, int64_t req_stride, const int32_t* seq_lens,
                                        const int32_t* q_row_offsets, int32_t batch, int64_t total_q_rows,
                                        int32_t max_q_rows, int64_t max_seq_len, float sm_scale,
                                        int32_t num_splits, uint16_t* out, void* stream) {
  // every argument check of ftkv_decode_attn, and its split geometry, before anything is enqueued
  ftkv::DecodeGeom geom;
  int st = ftkv::decode_validate(pool, num_q_heads, q, req_to_slot, req_stride, seq_lens, q_row_offsets, batch,
                                 total_q_rows, max_q_rows, max_seq_len, sm_scale, 0, num_splits, 0u, nullptr, 0,
                                 out, false, &geom);
  if (st != FTKV_OK || geom.empty) return st;
  if (geom.need > FTKV_NOALLOC_SCRATCH_BYTES) return FTKV_ERR_WORKSPACE;  // beyond the static maximum
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != FTKV_OK) return st;
  // scratch layout of this call (that of ftkv_decode_attn's workspace):
  // [partial accumulators | partial (max, sum) | arrival counters], 256-byte aligned parts
  const int64_t parts = geom.parts;
  const int64_t ctr_off = round256(parts * pool->head_dim * 4) + round256(parts * 2 * 4);
  const int64_t ctr_bytes = round256((static_cast<int64_t>(batch) * pool->num_kv_heads + 2) * 4);
  if (cudaMemsetAsync(static_cast<unsigned char*>(scratch) + ctr_off, 0, static_cast<size_t>(ctr_bytes),
                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FTKV_ERR_CUDA;
  return ftkv_decode_attn(pool, num_q_heads, q, req_to_slot, req_stride, seq_lens, q_row_offsets, batch,
                          total_q_rows, max_q_rows, max_seq_len, sm_scale, 0, static_cast<int32_t>(geom.splits),
                          0u, scratch, FTKV_NOALLOC_SCRATCH_BYTES, out, stream);
}
