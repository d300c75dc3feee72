/*
 * ftkv_oracle.c -- plain, slow CPU oracle for the FP8 (E4M3FN) per-token/per-head KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package smoke check and the benchmark's
 * CPU-baseline arm may load this library.  It shares no code, header, table or constant with the
 * CUDA path; the two meet only through the seeded synthetic inputs.
 *
 * Sources (the method as the pages describe it):
 *   [#853]  FreeToken PR #853 "opt-in FP8 KV cache (R9700)"
 *           - "What changes": each physical K/V row holds E4M3 codes as bytes plus its own FP32
 *             scale; prefill rebuilds historical FP8 rows into one shared BF16 workspace per layer
 *             while the current chunk stays BF16.
 *           - "Validation": byte accounting at 33,059 rows (BF16 KV, FP8 codes+scales, one
 *             workspace).
 *           - "Follow-up model/workload search": bytes/token BF16 vs FP8; every new K/V row is
 *             quantized on write and the per-row FP32 scales are loaded during attention.
 *   [#897]  FreeToken PR #897 "perf(attention): add packed fp8 kv reads on gfx1201"
 *           - opening description: codes are converted and used as BF16 for the attention math.
 *           - "Fresh R9700 stage-1 A/B": split-K decode (stage 1 + merge), reference = CPU FP8
 *             dequantization followed by attention.
 *           - "Regression and CUDA isolation": every finite E4M3FN value, signed zero included,
 *             must survive bit-for-bit.
 *   [#280]  FreeToken issue #280 "Feature Request: opt-in FP8 KV-cache support ..."
 *           - "Proof of concept" / limitations: E4M3 storage with dynamic per-token, per-KV-head
 *             FP32 scales.
 *   The absmax/448 scale and the saturating round-to-nearest-even encode are the plainest reading
 *   of "dynamic per-token/per-KV-head scale" for E4M3FN (largest finite magnitude 448); the
 *   readings taken where the pages are silent are listed in the design notes.
 *
 * Precision: attention is evaluated in IEEE double from the exactly dequantized values.  The store
 * and reconstruct steps use the FP32 operations the row format implies (one FP32 division, one
 * FP32 product, round-to-nearest-even to BF16).  Compile with -ffp-contract=off so no FMA
 * contraction changes an FP32 result.
 *
 * Parallelism: OpenMP `parallel for` over independent outputs only; no arithmetic is reordered.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------------------------ */
/* E4M3FN codec                                                                                */
/* ------------------------------------------------------------------------------------------ */

/* Decode one E4M3FN byte (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no
 * infinities, NaN only for exponent 15 with mantissa 7).  Written out from the format's
 * definition; [#897 "Regression and CUDA isolation"] requires every finite code to survive. */
double ftkv_oracle_e4m3_decode(uint8_t c) {
  int s = (c >> 7) & 1;
  int e = (c >> 3) & 15;
  int m = c & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);          /* subnormal: 2^-6 * m/8 */
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7); /* normal: 2^(e-7) * (1 + m/8) */
  return s ? -mag : mag;
}

/* The 127 non-negative finite magnitudes, ascending: entry i is the value of code i; and the value
 * of every code (g_dec), both filled from the closed form above. */
static double g_mag[127];
static double g_dec[256];
static int g_mag_ready = 0;

static void init_mag_table(void) {
  if (g_mag_ready) return;
  for (int i = 0; i < 127; i++) g_mag[i] = ftkv_oracle_e4m3_decode((uint8_t)i);
  for (int i = 0; i < 256; i++) g_dec[i] = ftkv_oracle_e4m3_decode((uint8_t)i);
  g_mag_ready = 1;
}

/* Encode one FP32 value to E4M3FN: round to the nearest finite E4M3 value, ties to the code with
 * an even mantissa (the code's least significant bit is 0), saturating to +-448.  NaN gives the
 * canonical code 0x7F; the sign bit is kept for every other input (so -0 -> 0x80). */
uint8_t ftkv_oracle_e4m3_encode(float x) {
  init_mag_table();
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a >= g_mag[126]) return sign | 126; /* +-448 and everything beyond it, +-Inf included */
  /* largest index lo with g_mag[lo] <= a (bisection over the ascending table) */
  int lo = 0, hi = 126;
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (g_mag[mid] <= a) lo = mid; else hi = mid;
  }
  /* candidates lo and lo+1 (= hi); the distances are exact in double */
  double dlo = a - g_mag[lo], dhi = g_mag[hi] - a;
  int code;
  if (dlo < dhi) code = lo;
  else if (dhi < dlo) code = hi;
  else code = (lo & 1) ? hi : lo; /* tie: even mantissa */
  return sign | (uint8_t)code;
}

void ftkv_oracle_e4m3_encode_array(const float* x, uint8_t* out, int64_t n) {
  init_mag_table();
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; i++) out[i] = ftkv_oracle_e4m3_encode(x[i]);
}

void ftkv_oracle_e4m3_decode_array(const uint8_t* c, double* out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = ftkv_oracle_e4m3_decode(c[i]);
}

/* ------------------------------------------------------------------------------------------ */
/* BF16 helpers                                                                                */
/* ------------------------------------------------------------------------------------------ */

static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round an FP32 value to BF16, nearest-even.  NaN maps to the quiet NaN 0x7FC0 (sign dropped). */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if (isnan(f)) return 0x7FC0;
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

uint16_t ftkv_oracle_f32_to_bf16(float f) { return f32_to_bf16_rne(f); }

/* ------------------------------------------------------------------------------------------ */
/* Quantize-on-write                                                                           */
/* ------------------------------------------------------------------------------------------ */

/* One (token, KV head) row of D BF16 values -> D codes + one FP32 scale.
 * [#853 "What changes"] each row carries its own FP32 scale; [#280 "Proof of concept"] the scale
 * is dynamic per token and KV head.  Reading: scale = absmax / 448 (FP32 division), code =
 * encode(x / scale) with an IEEE FP32 division; an all-zero row keeps scale 0 and divides by 1.
 * absmax ignores NaN (IEEE maxNum) and starts from +0. */
static void quantize_row(const uint16_t* x, int D, uint8_t* codes, float* scale) {
  float amax = 0.0f;
  for (int d = 0; d < D; d++) amax = fmaxf(amax, fabsf(bf16_to_f32(x[d])));
  float s = amax / 448.0f;
  float div = (s == 0.0f) ? 1.0f : s;
  for (int d = 0; d < D; d++) {
    float q = bf16_to_f32(x[d]) / div; /* one rounded FP32 quotient */
    codes[d] = ftkv_oracle_e4m3_encode(q);
  }
  *scale = s;
}

/* Store T new tokens: K/V BF16 [T][Hkv][D] into pool rows slots[t].
 * Pool layout: codes [num_rows][Hkv][D] bytes, scales [num_rows][Hkv] FP32.
 * [#853 "Follow-up model/workload search"]: each new K/V row is quantized when written. */
int ftkv_oracle_store_quant(const uint16_t* k, const uint16_t* v, const int32_t* slots, int64_t T,
                            int Hkv, int D, uint8_t* k_codes, uint8_t* v_codes, float* k_scales,
                            float* v_scales, int64_t num_rows) {
  init_mag_table();
  for (int64_t t = 0; t < T; t++)
    if (slots[t] < 0 || slots[t] >= num_rows) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; t++) {
    int64_t row = slots[t];
    for (int h = 0; h < Hkv; h++) {
      quantize_row(k + (t * Hkv + h) * D, D, k_codes + (row * Hkv + h) * D, k_scales + row * Hkv + h);
      quantize_row(v + (t * Hkv + h) * D, D, v_codes + (row * Hkv + h) * D, v_scales + row * Hkv + h);
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Reconstruct historical rows into the BF16 workspace                                         */
/* ------------------------------------------------------------------------------------------ */

/* ws[i][h][d] = bf16_rne( float(decode(code[slots[i]][h][d])) * scale[slots[i]][h] ).
 * [#853 "What changes"]: historical FP8 rows are rebuilt once per layer into one shared BF16
 * workspace.  Reading: the workspace is in logical order (row i of the workspace holds the
 * i-th historical token), the product is one FP32 multiplication, then round-to-nearest-even. */
int ftkv_oracle_reconstruct(const uint8_t* k_codes, const uint8_t* v_codes, const float* k_scales,
                            const float* v_scales, int64_t num_rows, int Hkv, int D,
                            const int32_t* slots, int64_t P, uint16_t* ws_k, uint16_t* ws_v) {
  init_mag_table();
  for (int64_t i = 0; i < P; i++)
    if (slots[i] < 0 || slots[i] >= num_rows) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < P; i++) {
    int64_t row = slots[i];
    for (int h = 0; h < Hkv; h++) {
      float sk = k_scales[row * Hkv + h], sv = v_scales[row * Hkv + h];
      for (int d = 0; d < D; d++) {
        float pk = (float)g_dec[k_codes[(row * Hkv + h) * D + d]] * sk;
        float pv = (float)g_dec[v_codes[(row * Hkv + h) * D + d]] * sv;
        ws_k[(i * Hkv + h) * D + d] = f32_to_bf16_rne(pk);
        ws_v[(i * Hkv + h) * D + d] = f32_to_bf16_rne(pv);
      }
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Attention (FP64)                                                                            */
/* ------------------------------------------------------------------------------------------ */

/* ---- decode over the FP8 pool, or over a BF16 pool ---- */
typedef struct {
  const uint8_t* codes;    /* FP8 pool: E4M3 codes [rows][Hkv][D] and FP32 scales [rows][Hkv] */
  const float* scales;
  const uint16_t* bf16;    /* BF16 pool: values [rows][Hkv][D] (codes == NULL) */
  const int32_t* slot_of;  /* logical key j -> pool row */
  int Hkv, D, h;
} pool_ctx;

/* Row j of one KV head as doubles: decode(code) * scale for the FP8 pool (exact in double), the BF16 value
 * itself for the BF16 pool (exact). */
static void pool_row(const pool_ctx* c, int64_t j, double* out) {
  int64_t row = c->slot_of[j];
  if (c->codes) {
    const uint8_t* code = c->codes + (row * c->Hkv + c->h) * c->D;
    double s = (double)c->scales[row * c->Hkv + c->h];
    for (int d = 0; d < c->D; d++) out[d] = g_dec[code[d]] * s;
  } else {
    const uint16_t* v = c->bf16 + (row * c->Hkv + c->h) * c->D;
    for (int d = 0; d < c->D; d++) out[d] = (double)bf16_to_f32(v[d]);
  }
}

/* Decode attention over a pool (shared by the FP8 and the BF16 entry points below).
 *   q:            BF16 [total_rows][Hq][D]
 *   req_to_slot:  int32 [B][req_stride]; key j of request b lives in pool row req_to_slot[b*stride+j]
 *   seq_lens:     int32 [B]; request b has seq_lens[b] keys (the new rows included)
 *   q_row_offsets int32 [B+1]; request b owns query rows [q_row_offsets[b], q_row_offsets[b+1])
 *   window:       0 = full attention; W >= 1 = sliding window: a row whose visible keys are 0 .. v-1
 *                 attends to keys max(0, v-W) .. v-1 (its own position included)
 *   out:          double [total_rows][Hq][D]
 *   abs_v:        if nonzero, accumulate |v^| instead of v^ (the attention-weighted magnitude of the
 *                 summed terms, used by the tests to size the rounding bound; not part of the method)
 * [#897 "Fresh R9700 stage-1 A/B"]: the reference is CPU FP8 dequantization followed by attention;
 * split-K is an evaluation order and does not appear here.  Multi-row decode (up to 8 rows per
 * request, [#897 opening description]) is causal within the rows; reading: row r of R rows sees
 * keys 0 .. n-R+r.  Query head i reads KV head i / (Hq/Hkv).  The sliding window is one of the
 * integration cases of [#897 "Regression and CUDA isolation"] ("odd sliding window"); its reading is the
 * usual one (the last W positions up to the query's own). */
static int decode_core(const uint8_t* k_codes, const uint8_t* v_codes, const float* k_scales,
                       const float* v_scales, const uint16_t* k_bf16, const uint16_t* v_bf16,
                       int64_t num_rows, int Hq, int Hkv, int D, const uint16_t* q, const int32_t* req_to_slot,
                       int64_t req_stride, const int32_t* seq_lens, const int32_t* q_row_offsets, int B,
                       double sm_scale, int64_t window, int abs_v, double* out) {
  init_mag_table();
  if (Hkv <= 0 || Hq % Hkv != 0 || window < 0) return -1;
  int G = Hq / Hkv;
  int64_t max_n = 0;
  for (int b = 0; b < B; b++) {
    if (seq_lens[b] < 0 || seq_lens[b] > req_stride) return -1;
    for (int64_t j = 0; j < seq_lens[b]; j++) {
      int32_t r = req_to_slot[b * req_stride + j];
      if (r < 0 || r >= num_rows) return -1;
    }
    if (seq_lens[b] > max_n) max_n = seq_lens[b];
  }
  int total = q_row_offsets[B];
  /* one task per (query row, head) */
  int64_t ntask = (int64_t)total * Hq;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (max_n > 0 ? max_n : 1));
    double* kv = (double*)malloc(sizeof(double) * D);
    double* qd = (double*)malloc(sizeof(double) * D);
#pragma omp for schedule(dynamic, 4)
    for (int64_t task = 0; task < ntask; task++) {
      int row = (int)(task / Hq), i = (int)(task % Hq);
      int b = 0;
      while (!(q_row_offsets[b] <= row && row < q_row_offsets[b + 1])) b++;
      int R = q_row_offsets[b + 1] - q_row_offsets[b];
      int r = row - q_row_offsets[b];
      int64_t visible = (int64_t)seq_lens[b] - R + r + 1;
      if (visible < 0) visible = 0;
      int64_t first = (window > 0 && visible > window) ? visible - window : 0;
      for (int d = 0; d < D; d++) qd[d] = (double)bf16_to_f32(q[((int64_t)row * Hq + i) * D + d]);
      pool_ctx kc = {k_codes, k_scales, k_bf16, req_to_slot + b * req_stride, Hkv, D, i / G};
      pool_ctx vc = {v_codes, v_scales, v_bf16, req_to_slot + b * req_stride, Hkv, D, i / G};
      double* o = out + ((int64_t)row * Hq + i) * D;
      for (int d = 0; d < D; d++) o[d] = 0.0;
      if (visible > first) {
        double m = -INFINITY;
        for (int64_t j = first; j < visible; j++) {
          pool_row(&kc, j, kv);
          double dot = 0.0;
          for (int d = 0; d < D; d++) dot += qd[d] * kv[d];
          s[j] = dot * sm_scale;
          if (s[j] > m) m = s[j];
        }
        double l = 0.0;
        for (int64_t j = first; j < visible; j++) {
          double p = exp(s[j] - m);
          l += p;
          pool_row(&vc, j, kv);
          for (int d = 0; d < D; d++) o[d] += p * (abs_v ? fabs(kv[d]) : kv[d]);
        }
        for (int d = 0; d < D; d++) o[d] /= l;
      }
    }
    free(s);
    free(kv);
    free(qd);
  }
  return 0;
}

/* Decode attention over the FP8 pool (codes [rows][Hkv][D], FP32 scales [rows][Hkv]). */
int ftkv_oracle_decode_attn(const uint8_t* k_codes, const uint8_t* v_codes, const float* k_scales,
                            const float* v_scales, int64_t num_rows, int Hq, int Hkv, int D,
                            const uint16_t* q, const int32_t* req_to_slot, int64_t req_stride,
                            const int32_t* seq_lens, const int32_t* q_row_offsets, int B,
                            double sm_scale, int64_t window, int abs_v, double* out) {
  if (!k_codes || !v_codes || !k_scales || !v_scales) return -1;
  return decode_core(k_codes, v_codes, k_scales, v_scales, NULL, NULL, num_rows, Hq, Hkv, D, q, req_to_slot,
                     req_stride, seq_lens, q_row_offsets, B, sm_scale, window, abs_v, out);
}

/* Decode attention over a BF16 pool (values [rows][Hkv][D]): the BF16 KV cache the FP8 format replaces
 * ([#853 "Follow-up model/workload search"]: 98,304 vs 50,688 bytes per token), same definition. */
int ftkv_oracle_decode_attn_bf16(const uint16_t* k, const uint16_t* v, int64_t num_rows, int Hq, int Hkv, int D,
                                 const uint16_t* q, const int32_t* req_to_slot, int64_t req_stride,
                                 const int32_t* seq_lens, const int32_t* q_row_offsets, int B, double sm_scale,
                                 int64_t window, int abs_v, double* out) {
  if (!k || !v) return -1;
  return decode_core(NULL, NULL, NULL, NULL, k, v, num_rows, Hq, Hkv, D, q, req_to_slot, req_stride, seq_lens,
                     q_row_offsets, B, sm_scale, window, abs_v, out);
}

/* ---- prefill over the BF16 workspace prefix plus the BF16 chunk ---- */
typedef struct {
  const uint16_t* prefix; /* [P][Hkv][D] */
  const uint16_t* chunk;  /* [C][Hkv][D] */
  int64_t P;
  int Hkv, D, h;
} cat_ctx;

/* Key/value j of the concatenation prefix (+) chunk for one KV head. */
static void cat_row(const cat_ctx* c, int64_t j, double* out) {
  const uint16_t* src = (j < c->P) ? c->prefix + (j * c->Hkv + c->h) * c->D
                                   : c->chunk + ((j - c->P) * c->Hkv + c->h) * c->D;
  for (int d = 0; d < c->D; d++) out[d] = (double)bf16_to_f32(src[d]);
}

/* Prefill (extend) attention for the current chunk.
 *   q, k_chunk, v_chunk: BF16 [C][Hq|Hkv][D];  ws_k, ws_v: BF16 [P][Hkv][D] (reconstructed prefix)
 *   rows: the chunk query indices to evaluate (n_rows of them; NULL = all C rows in order)
 *   out:  double [n_rows][Hq][D]
 *   abs_v: if nonzero, accumulate |v| instead of v (test helper, as for decode)
 * [#853 "What changes"]: keys/values are the rebuilt BF16 prefix followed by the BF16 current
 * chunk; chunk query t sees the whole prefix and chunk keys 0..t (causal). */
int ftkv_oracle_prefill_attn(int Hq, int Hkv, int D, const uint16_t* q, const uint16_t* k_chunk,
                             const uint16_t* v_chunk, int64_t C, const uint16_t* ws_k,
                             const uint16_t* ws_v, int64_t P, double sm_scale, const int64_t* rows,
                             int64_t n_rows, int abs_v, double* out) {
  if (Hkv <= 0 || Hq % Hkv != 0) return -1;
  int G = Hq / Hkv;
  if (rows)
    for (int64_t r = 0; r < n_rows; r++)
      if (rows[r] < 0 || rows[r] >= C) return -1;
  int64_t ntask = n_rows * Hq;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (P + C > 0 ? P + C : 1));
    double* kv = (double*)malloc(sizeof(double) * D);
    double* qd = (double*)malloc(sizeof(double) * D);
#pragma omp for schedule(dynamic, 4)
    for (int64_t task = 0; task < ntask; task++) {
      int64_t ri = task / Hq;
      int i = (int)(task % Hq);
      int64_t t = rows ? rows[ri] : ri;
      for (int d = 0; d < D; d++) qd[d] = (double)bf16_to_f32(q[(t * Hq + i) * D + d]);
      cat_ctx kc = {ws_k, k_chunk, P, Hkv, D, i / G};
      cat_ctx vc = {ws_v, v_chunk, P, Hkv, D, i / G};
      double* o = out + (ri * Hq + i) * D;
      int64_t n = P + t + 1;
      for (int d = 0; d < D; d++) o[d] = 0.0;
      double m = -INFINITY;
      for (int64_t j = 0; j < n; j++) {
        cat_row(&kc, j, kv);
        double dot = 0.0;
        for (int d = 0; d < D; d++) dot += qd[d] * kv[d];
        s[j] = dot * sm_scale;
        if (s[j] > m) m = s[j];
      }
      double l = 0.0;
      for (int64_t j = 0; j < n; j++) {
        double p = exp(s[j] - m);
        l += p;
        cat_row(&vc, j, kv);
        for (int d = 0; d < D; d++) o[d] += p * (abs_v ? fabs(kv[d]) : kv[d]);
      }
      for (int d = 0; d < D; d++) o[d] /= l;
    }
    free(s);
    free(kv);
    free(qd);
  }
  return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Byte accounting                                                                             */
/* ------------------------------------------------------------------------------------------ */

/* [#853 "Validation"] and "Follow-up model/workload search": persistent KV bytes for `rows`
 * physical rows over `layers` layers.
 *   BF16 KV      = rows * layers * Hkv * D * 2 bytes * 2 tensors
 *   FP8 KV       = rows * layers * (2 tensors * Hkv * D code bytes + 2 tensors * Hkv * 4 scale bytes)
 *   workspace    = rows * Hkv * D * 2 bytes * 2 tensors (one layer, BF16, shared)            */
void ftkv_oracle_pool_bytes(int64_t rows, int64_t layers, int64_t Hkv, int64_t D, int64_t* bf16_bytes,
                            int64_t* fp8_bytes, int64_t* workspace_bytes) {
  *bf16_bytes = rows * layers * Hkv * D * 2 * 2;
  *fp8_bytes = rows * layers * (2 * Hkv * D + 2 * Hkv * 4);
  *workspace_bytes = rows * Hkv * D * 2 * 2;
}

/* ------------------------------------------------------------------------------------------ */
void ftkv_oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int ftkv_oracle_get_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
