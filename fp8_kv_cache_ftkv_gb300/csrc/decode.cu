// decode.cu -- split-K decode attention over the FP8 (E4M3FN) pool: what it computes, and which kernel runs it.
//
// What it computes (FreeToken PR #897, opening description and "Fresh R9700 stage-1 A/B"): for a request with
// n keys and a BF16 query row, per query head i (KV head h = i / G)
//     s_j = (q . k^_j) * sm_scale,   k^_j = decode(codeK_j) * scaleK_j,   v^_j likewise,
//     o   = sum_j softmax(s)_j v^_j,
// with split-K over the keys: each CTA covers one slice of the keys and writes a partial (max, sum,
// accumulator); the last slice of a (request, KV head) to finish merges them in the same call.  Multi-row
// decode: row r of a request's R rows sees keys 0 .. n-R+r (or the last W of them with a sliding window).
//
// Both kernels read the stored codes and scales directly (no dequantized copy of the pool), run QK^T on the
// FP8 tensor cores with the query in two E4M3 pieces and PV on FP16 tensor cores with the V scale folded into
// the probabilities, with a lazy softmax maximum and a lazy power-of-two unit for the FP16 operands:
//  * single-row batches (max_q_rows = 1): decode_tok.cu -- a CTA covers every KV head of a token (one
//    contiguous run of the pool row), mma.sync on 16-key blocks, two CTAs per SM;
//  * multi-row batches: decode_mr.cu -- a CTA covers one KV head of a request's key slice, tcgen05 MMAs on
//    128-key tiles with S, O and P in tensor memory, one CTA per SM.
#include "ftkv_internal.h"

namespace ftkv {

int decode_ctas_per_sm(int max_q_rows) {
  // the token-major single-row kernel fits two CTAs per SM; the multi-row kernel is shared-memory bound at one
  return max_q_rows <= 1 ? 2 : 1;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  if (a.max_q_rows <= 1) return launch_decode_tok(a, s);
  return launch_decode_mr(a, s);
}

}  // namespace ftkv
