/*
 * kvq_oracle.c — plain CPU oracle of the rotated INT2 KV-cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, the package's smoke() check and the
 * benchmark's CPU-baseline leg may load this library.  The product path
 * (libkvq.so and its binding) never calls it and shares no code with it.
 *
 * It is written for a reader checking it by eye against the method's
 * description, not for speed: one vector, one token, one head at a time, in the
 * order the method states its steps.  Floating point:
 *   - attention is computed in float64 on the dequantised cache;
 *   - the quantiser follows an explicit fp32 operation sequence (the method does
 *     not fix the precision; this fixed sequence makes the stored codes exactly
 *     reproducible).  Build with -ffp-contract=off so that no multiply-add is
 *     fused except where fmaf() is written.
 *
 * Sources (page title, then section):
 *   [OptR] "Output-Aware Rotation for INT2 KV-Cache Quantization", pith.science
 *          review of arXiv 2608.02691.
 *   - "What carries the argument", mechanism (2): keys are centred, k -> k - mu,
 *     before rotation and quantisation; attention-equivalent.
 *   - same section, mechanism (3): rotation, clipping, grouping, rounding,
 *     dequantisation and inverse rotation form the quantised path.
 *   - "Assumptions & free parameters": clipping ratios c_K = 0.96, c_V = 0.92;
 *     separate key and value rotation corrections (A_K, A_V).
 *   - "If this is right", third item: the paged KV-cache layout is preserved and
 *     value-side rotations fold into W_V / W_O.
 * Readings where the pages are silent (asymmetric INT2, one group of 128 along
 * head_dim, fp16 scale/zero, clip scales the group max and min toward zero,
 * round half to even, row-vector rotation) are stated at each function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define PAGE 16
#define DIM 128
#define INT2_REC 1152
#define BF16_REC 8192

/* ------------------------------------------------------------------------- */
/* Number formats (IEEE 754 binary16 and bfloat16), written from the formats'  */
/* definitions.                                                              */
/* ------------------------------------------------------------------------- */

static uint32_t f32_bits(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }
static float bits_f32(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }

/* binary16 -> binary32, exact. */
float kvqo_f16_to_f32(uint16_t h) {
  uint32_t sign = (uint32_t)(h >> 15) & 1u;
  uint32_t e = (uint32_t)(h >> 10) & 0x1fu;
  uint32_t m = (uint32_t)h & 0x3ffu;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24);             /* subnormal: m * 2^-24 */
  } else if (e == 31) {
    if (m) return bits_f32(0x7fc00000u | (sign << 31));
    v = INFINITY;
  } else {
    v = ldexp((double)(1024 + m), (int)e - 25);  /* (1 + m/1024) * 2^(e-15) */
  }
  return (float)(sign ? -v : v);
}

/* binary32 -> binary16, round to nearest, ties to even.  Written on the
 * exact value: find the binary16 neighbours of |x| and pick the nearer one,
 * the even one on a tie.  Overflow beyond the largest finite value rounds to
 * infinity when |x| >= 65520 (the midpoint between 65504 and 2^16). */
uint16_t kvqo_f32_to_f16(float x) {
  uint32_t u = f32_bits(x);
  uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  if (isnan(x)) return (uint16_t)(sign | 0x7e00u);
  double a = fabs((double)x);
  if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u);
  /* spacing of binary16 numbers around a: 2^-24 below 2^-14, else 2^(E-10) */
  int E;
  if (a < ldexp(1.0, -14)) {
    E = -14;
  } else {
    E = (int)floor(log2(a));
    /* guard against log2 rounding at exact powers of two */
    if (ldexp(1.0, E) > a) E -= 1;
    if (ldexp(1.0, E + 1) <= a) E += 1;
  }
  double ulp = ldexp(1.0, E - 10);
  double q = a / ulp;                 /* exact: a is a binary32, ulp a power of two */
  double lo = floor(q);
  double frac = q - lo;
  double n;
  if (frac > 0.5) n = lo + 1.0;
  else if (frac < 0.5) n = lo;
  else n = (fmod(lo, 2.0) == 0.0) ? lo : lo + 1.0;
  double r = n * ulp;                 /* the rounded magnitude */
  if (r >= 65536.0) return (uint16_t)(sign | 0x7c00u);
  /* encode r */
  if (r < ldexp(1.0, -14)) {
    uint16_t m = (uint16_t)(r / ldexp(1.0, -24));
    return (uint16_t)(sign | m);
  }
  int Er = (int)floor(log2(r));
  if (ldexp(1.0, Er) > r) Er -= 1;
  if (ldexp(1.0, Er + 1) <= r) Er += 1;
  uint16_t m = (uint16_t)(r / ldexp(1.0, Er - 10) - 1024.0);
  return (uint16_t)(sign | (uint16_t)((Er + 15) << 10) | m);
}

/* bfloat16 -> binary32, exact (bfloat16 is the top half of a binary32). */
float kvqo_bf16_to_f32(uint16_t b) { return bits_f32((uint32_t)b << 16); }

/* ------------------------------------------------------------------------- */
/* Quantiser                                                                 */
/* ------------------------------------------------------------------------- */

/* Quantise one vector x (bf16 bit patterns, D elements) of one token and head.
 * [OptR] "What carries the argument": centre (keys only) -> rotate -> clip ->
 * group -> round.  Readings: one group = the whole vector (128 elements); the
 * clip ratio c scales the group max and min toward zero; asymmetric grid with
 * scale s = (c*max - c*min)/3 and zero z = c*min, both stored as fp16 and the
 * codes computed against the stored (fp16-rounded) s and z; round half to even;
 * a group whose stored scale is 0 gets all codes 0.  The rotation is applied to
 * the row vector, r_i = sum_j c_j R[j][i], as a sequential fp32 fmaf chain in
 * j order.
 *   mu      : key mean (D floats) or NULL for values.
 *   R       : D x D fp32, R[j*D + i].
 *   codes   : out, D bytes in 0..3.
 *   s16,z16 : out, fp16 bit patterns.
 *   r_out   : optional out, the rotated fp32 vector.
 *   t_out   : optional out, the pre-rounding values (r_i - z) / s (0 if s == 0). */
void kvqo_quantize(const uint16_t* x, const float* mu, const float* R, int D, float clip,
                   uint8_t* codes, uint16_t* s16, uint16_t* z16, float* r_out, float* t_out) {
  float* c = (float*)malloc(sizeof(float) * (size_t)D);
  float* r = (float*)malloc(sizeof(float) * (size_t)D);
  /* centre (keys) */
  for (int j = 0; j < D; ++j) {
    float xf = kvqo_bf16_to_f32(x[j]);
    c[j] = mu ? (xf - mu[j]) : xf;
  }
  /* rotate: row vector times R, fixed-order fp32 fused multiply-add chain */
  for (int i = 0; i < D; ++i) {
    float acc = 0.0f;
    for (int j = 0; j < D; ++j) acc = fmaf(c[j], R[(size_t)j * D + i], acc);
    r[i] = acc;
  }
  /* group statistics (one group = the whole vector) */
  float mx = r[0], mn = r[0];
  for (int i = 1; i < D; ++i) {
    mx = fmaxf(mx, r[i]);
    mn = fminf(mn, r[i]);
  }
  /* clip toward zero, asymmetric scale and zero */
  float mxc = clip * mx;
  float mnc = clip * mn;
  float s32 = (mxc - mnc) / 3.0f;
  uint16_t sh = kvqo_f32_to_f16(s32);
  uint16_t zh = kvqo_f32_to_f16(mnc);
  float s = kvqo_f16_to_f32(sh);
  float z = kvqo_f16_to_f32(zh);
  for (int i = 0; i < D; ++i) {
    if (s == 0.0f) {
      codes[i] = 0;
      if (t_out) t_out[i] = 0.0f;
    } else {
      float t = (r[i] - z) / s;
      float k = fminf(fmaxf(rintf(t), 0.0f), 3.0f);
      codes[i] = (uint8_t)k;
      if (t_out) t_out[i] = t;
    }
    if (r_out) r_out[i] = r[i];
  }
  *s16 = sh;
  *z16 = zh;
  free(c);
  free(r);
}

/* ------------------------------------------------------------------------- */
/* Page records (the library's byte layout; see include/kvq.h)               */
/* ------------------------------------------------------------------------- */

/* Byte offset and bit shift of the 2-bit code of (slot tau, element d) in an
 * INT2 record; which = 0 keys, 1 values.  Transcribes the header's formulas. */
void kvqo_int2_locate(int which, int tau, int d, int* byte, int* shift) {
  int lane, word, bit;
  if (which == 0) {
    int w = d >> 4, r = d & 15, h = r >> 3, t = (r >> 1) & 3, e = r & 1;
    lane = 4 * (tau & 7) + t;
    word = 2 * (tau >> 3) + h;
    bit = 16 * e + 2 * w;
    *byte = 16 * lane + 4 * word + (bit >> 3);
  } else {
    int m = d >> 4, r = d & 15, g = r & 7, dh = r >> 3;
    int t = (tau & 7) >> 1, e = tau & 1, th = tau >> 3;
    lane = 4 * g + t;
    word = 2 * th + dh;
    bit = 16 * e + 2 * m;
    *byte = 512 + 16 * lane + 4 * word + (bit >> 3);
  }
  *shift = bit & 7;
}

/* Byte offset of the fp16 scale of (slot tau); the zero follows at +2. */
int kvqo_int2_meta_offset(int which, int tau) {
  return 1024 + 16 * (tau & 7) + (which ? 8 : 0) + 4 * (tau >> 3);
}

void kvqo_int2_store(uint8_t* rec, int which, int tau, const uint8_t* codes, uint16_t s16,
                     uint16_t z16) {
  for (int d = 0; d < DIM; ++d) {
    int byte, shift;
    kvqo_int2_locate(which, tau, d, &byte, &shift);
    rec[byte] = (uint8_t)((rec[byte] & ~(3u << shift)) | ((codes[d] & 3u) << shift));
  }
  int o = kvqo_int2_meta_offset(which, tau);
  rec[o + 0] = (uint8_t)(s16 & 0xff);
  rec[o + 1] = (uint8_t)(s16 >> 8);
  rec[o + 2] = (uint8_t)(z16 & 0xff);
  rec[o + 3] = (uint8_t)(z16 >> 8);
}

void kvqo_int2_load(const uint8_t* rec, int which, int tau, uint8_t* codes, uint16_t* s16,
                    uint16_t* z16) {
  for (int d = 0; d < DIM; ++d) {
    int byte, shift;
    kvqo_int2_locate(which, tau, d, &byte, &shift);
    codes[d] = (uint8_t)((rec[byte] >> shift) & 3u);
  }
  int o = kvqo_int2_meta_offset(which, tau);
  *s16 = (uint16_t)(rec[o] | (rec[o + 1] << 8));
  *z16 = (uint16_t)(rec[o + 2] | (rec[o + 3] << 8));
}

/* Byte offset of the bf16 element (slot tau, element d) in a BF16 record. */
int kvqo_bf16_locate(int which, int tau, int d) {
  if (which == 0) {
    int w = d >> 4, r = d & 15, h = r >> 3, t = (r >> 1) & 3, e = r & 1;
    int lane = 4 * (tau & 7) + t, reg = (tau >> 3) + 2 * h;
    return 512 * w + 16 * lane + 4 * reg + 2 * e;
  } else {
    int m = d >> 4, r = d & 15, g = r & 7, dh = r >> 3;
    int t = (tau & 7) >> 1, e = tau & 1, th = tau >> 3;
    int lane = 4 * g + t, reg = 2 * th + dh;
    return 4096 + 512 * m + 16 * lane + 4 * reg + 2 * e;
  }
}

/* ------------------------------------------------------------------------- */
/* Append                                                                    */
/* ------------------------------------------------------------------------- */

/* Page record of (sequence b, position p, kv head) or NULL if the page table
 * entry or position is out of range.  [OptR] "If this is right", third item:
 * the paged layout — a page table maps position / 16 to a pool page. */
static uint8_t* record_of(uint8_t* pool, size_t rec_bytes, int Hkv, int num_pool_pages,
                          const int32_t* page_table, int max_pages, int b, int p, int kv) {
  if (p < 0 || p >= max_pages * PAGE) return NULL;
  int32_t page = page_table[(size_t)b * max_pages + p / PAGE];
  if (page < 0 || page >= num_pool_pages) return NULL;
  return pool + ((size_t)page * Hkv + kv) * rec_bytes;
}

/* Quantise and store n tokens (all KV heads, keys and values).
 *   R  : fp32 [2][Hkv][D][D] (keys then values), mu : fp32 [Hkv][D].
 * Returns the number of tokens skipped for a bad sequence, position or page. */
int kvqo_append_int2(uint8_t* pool, int num_pool_pages, int Hkv, const uint16_t* K,
                     const uint16_t* V, const int32_t* seq_idx, const int32_t* positions, int n,
                     const int32_t* page_table, int batch, int max_pages, const float* R,
                     const float* mu, float clip_k, float clip_v) {
  int skipped = 0;
  uint8_t codes[DIM];
  uint16_t s16, z16;
  for (int i = 0; i < n; ++i) {
    int b = seq_idx[i];
    if (b < 0 || b >= batch) { ++skipped; continue; }
    for (int kv = 0; kv < Hkv; ++kv) {
      uint8_t* rec = record_of(pool, INT2_REC, Hkv, num_pool_pages, page_table, max_pages, b,
                               positions[i], kv);
      if (!rec) { ++skipped; break; }
      int tau = positions[i] % PAGE;
      const float* RK = R + ((size_t)0 * Hkv + kv) * DIM * DIM;
      const float* RV = R + ((size_t)1 * Hkv + kv) * DIM * DIM;
      kvqo_quantize(K + ((size_t)i * Hkv + kv) * DIM, mu + (size_t)kv * DIM, RK, DIM, clip_k,
                    codes, &s16, &z16, NULL, NULL);
      kvqo_int2_store(rec, 0, tau, codes, s16, z16);
      kvqo_quantize(V + ((size_t)i * Hkv + kv) * DIM, NULL, RV, DIM, clip_v, codes, &s16, &z16,
                    NULL, NULL);
      kvqo_int2_store(rec, 1, tau, codes, s16, z16);
    }
  }
  return skipped;
}

/* Store n tokens unchanged into the BF16 comparison cache. */
int kvqo_append_bf16(uint8_t* pool, int num_pool_pages, int Hkv, const uint16_t* K,
                     const uint16_t* V, const int32_t* seq_idx, const int32_t* positions, int n,
                     const int32_t* page_table, int batch, int max_pages) {
  int skipped = 0;
  for (int i = 0; i < n; ++i) {
    int b = seq_idx[i];
    if (b < 0 || b >= batch) { ++skipped; continue; }
    for (int kv = 0; kv < Hkv; ++kv) {
      uint8_t* rec = record_of(pool, BF16_REC, Hkv, num_pool_pages, page_table, max_pages, b,
                               positions[i], kv);
      if (!rec) { ++skipped; break; }
      int tau = positions[i] % PAGE;
      for (int d = 0; d < DIM; ++d) {
        uint16_t k = K[((size_t)i * Hkv + kv) * DIM + d];
        uint16_t v = V[((size_t)i * Hkv + kv) * DIM + d];
        int ok = kvqo_bf16_locate(0, tau, d), ov = kvqo_bf16_locate(1, tau, d);
        rec[ok] = (uint8_t)(k & 0xff); rec[ok + 1] = (uint8_t)(k >> 8);
        rec[ov] = (uint8_t)(v & 0xff); rec[ov + 1] = (uint8_t)(v >> 8);
      }
    }
  }
  return skipped;
}

/* ------------------------------------------------------------------------- */
/* Dequantisation and attention                                              */
/* ------------------------------------------------------------------------- */

/* Dequantise (sequence b, positions [start, start+len)) to fp32 in the rotated
 * basis: x~ = fmaf(code, s, z).  Out: [len][Hkv][D]; either may be NULL.
 * Returns the number of positions skipped (bad page or position). */
int kvqo_dequant_int2(const uint8_t* pool, int num_pool_pages, int Hkv,
                      const int32_t* page_table, int max_pages, int b, int start, int len,
                      float* K_out, float* V_out) {
  int skipped = 0;
  uint8_t codes[DIM];
  uint16_t s16, z16;
  for (int i = 0; i < len; ++i) {
    int p = start + i;
    for (int kv = 0; kv < Hkv; ++kv) {
      const uint8_t* rec = record_of((uint8_t*)pool, INT2_REC, Hkv, num_pool_pages, page_table,
                                     max_pages, b, p, kv);
      if (!rec) { ++skipped; break; }
      for (int which = 0; which < 2; ++which) {
        float* o = which ? V_out : K_out;
        if (!o) continue;
        kvqo_int2_load(rec, which, p % PAGE, codes, &s16, &z16);
        float s = kvqo_f16_to_f32(s16), z = kvqo_f16_to_f32(z16);
        for (int d = 0; d < DIM; ++d)
          o[((size_t)i * Hkv + kv) * DIM + d] = fmaf((float)codes[d], s, z);
      }
    }
  }
  return skipped;
}

/* Row vector times matrix in float64: y_i = sum_j x_j M[j][i]. */
void kvqo_rotate_f64(const double* x, const float* M, int D, double* y) {
  for (int i = 0; i < D; ++i) {
    double acc = 0.0;
    for (int j = 0; j < D; ++j) acc += x[j] * (double)M[(size_t)j * D + i];
    y[i] = acc;
  }
}

/* Row vector times the transpose, in float64: y_i = sum_j x_j M[i][j]. */
void kvqo_rotate_t_f64(const double* x, const float* M, int D, double* y) {
  for (int i = 0; i < D; ++i) {
    double acc = 0.0;
    for (int j = 0; j < D; ++j) acc += x[j] * (double)M[(size_t)i * D + j];
    y[i] = acc;
  }
}

/* Softmax attention of one query over T keys/values, float64.
 *   q : [D], keys : [T][D], values : [T][D], out : [D].
 * logit_t = scale * q . k_t ; p = softmax(logit) ; out = sum_t p_t v_t.
 * T == 0 gives out = 0. */
void kvqo_attend_f64(const double* q, const double* keys, const double* values, int T, int D,
                     double scale, double* out) {
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (T <= 0) return;
  double* logit = (double*)malloc(sizeof(double) * (size_t)T);
  double mx = -INFINITY;
  for (int t = 0; t < T; ++t) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += q[d] * keys[(size_t)t * D + d];
    logit[t] = scale * acc;
    if (logit[t] > mx) mx = logit[t];
  }
  double sum = 0.0;
  for (int t = 0; t < T; ++t) {
    logit[t] = exp(logit[t] - mx);
    sum += logit[t];
  }
  for (int t = 0; t < T; ++t) {
    double p = logit[t] / sum;
    for (int d = 0; d < D; ++d) out[d] += p * values[(size_t)t * D + d];
  }
  free(logit);
}

/* INT2 decode for one (sequence b, query head hq), float64, over the pool bytes.
 * [OptR] "What carries the argument": the query meets the rotated, centred
 * keys (q_rot = q R_K, so q_rot . (k - mu) R_K = q . (k - mu)); the value path
 * ends with the inverse rotation o = o_rot R_V^T, left out when out_rotated is
 * set ("If this is right", third item: folded into W_V / W_O).
 *   q   : bf16 [D] of this head;  R : fp32 [2][Hkv][D][D].
 *   out : [D].  Returns the number of positions skipped (bad page). */
int kvqo_decode_int2_head(const uint8_t* pool, int num_pool_pages, int H, int Hkv,
                          const uint16_t* q, const int32_t* page_table, int max_pages, int b,
                          int seq_len, int hq, const float* R, double sm_scale, int out_rotated,
                          double* out) {
  int G = H / Hkv, kv = hq / G, skipped = 0;
  const float* RK = R + ((size_t)0 * Hkv + kv) * DIM * DIM;
  const float* RV = R + ((size_t)1 * Hkv + kv) * DIM * DIM;
  double qd[DIM], qrot[DIM], orot[DIM];
  for (int d = 0; d < DIM; ++d) qd[d] = (double)kvqo_bf16_to_f32(q[d]);
  kvqo_rotate_f64(qd, RK, DIM, qrot);
  double* keys = (double*)calloc((size_t)(seq_len > 0 ? seq_len : 1) * DIM, sizeof(double));
  double* vals = (double*)calloc((size_t)(seq_len > 0 ? seq_len : 1) * DIM, sizeof(double));
  int T = 0;
  uint8_t codes[DIM];
  uint16_t s16, z16;
  for (int p = 0; p < seq_len; ++p) {
    const uint8_t* rec = record_of((uint8_t*)pool, INT2_REC, Hkv, num_pool_pages, page_table,
                                   max_pages, b, p, kv);
    if (!rec) { ++skipped; continue; }
    kvqo_int2_load(rec, 0, p % PAGE, codes, &s16, &z16);
    double s = kvqo_f16_to_f32(s16), z = kvqo_f16_to_f32(z16);
    for (int d = 0; d < DIM; ++d) keys[(size_t)T * DIM + d] = (double)codes[d] * s + z;
    kvqo_int2_load(rec, 1, p % PAGE, codes, &s16, &z16);
    s = kvqo_f16_to_f32(s16);
    z = kvqo_f16_to_f32(z16);
    for (int d = 0; d < DIM; ++d) vals[(size_t)T * DIM + d] = (double)codes[d] * s + z;
    ++T;
  }
  kvqo_attend_f64(qrot, keys, vals, T, DIM, sm_scale, orot);
  if (out_rotated) {
    for (int d = 0; d < DIM; ++d) out[d] = orot[d];
  } else {
    kvqo_rotate_t_f64(orot, RV, DIM, out);
  }
  free(keys);
  free(vals);
  return skipped;
}

/* BF16 comparison decode for one (b, hq): plain float64 attention over the
 * stored bf16 keys and values with the unrotated query. */
int kvqo_decode_bf16_head(const uint8_t* pool, int num_pool_pages, int H, int Hkv,
                          const uint16_t* q, const int32_t* page_table, int max_pages, int b,
                          int seq_len, int hq, double sm_scale, double* out) {
  int G = H / Hkv, kv = hq / G, skipped = 0;
  double qd[DIM];
  for (int d = 0; d < DIM; ++d) qd[d] = (double)kvqo_bf16_to_f32(q[d]);
  double* keys = (double*)calloc((size_t)(seq_len > 0 ? seq_len : 1) * DIM, sizeof(double));
  double* vals = (double*)calloc((size_t)(seq_len > 0 ? seq_len : 1) * DIM, sizeof(double));
  int T = 0;
  for (int p = 0; p < seq_len; ++p) {
    const uint8_t* rec = record_of((uint8_t*)pool, BF16_REC, Hkv, num_pool_pages, page_table,
                                   max_pages, b, p, kv);
    if (!rec) { ++skipped; continue; }
    for (int d = 0; d < DIM; ++d) {
      int ok = kvqo_bf16_locate(0, p % PAGE, d), ov = kvqo_bf16_locate(1, p % PAGE, d);
      keys[(size_t)T * DIM + d] = kvqo_bf16_to_f32((uint16_t)(rec[ok] | (rec[ok + 1] << 8)));
      vals[(size_t)T * DIM + d] = kvqo_bf16_to_f32((uint16_t)(rec[ov] | (rec[ov + 1] << 8)));
    }
    ++T;
  }
  kvqo_attend_f64(qd, keys, vals, T, DIM, sm_scale, out);
  free(keys);
  free(vals);
  return skipped;
}

/* Decode with a BF16 window, for one (b, hq), float64.  [OptR] "Assumptions &
 * free parameters": a BF16 window of sink tokens (the first ones) and recent
 * tokens (the last ones) is kept at full precision; the rest of the context is
 * read from the INT2 cache.  Positions [0, sink) and [len - recent, len) come
 * from the BF16 pool (plain keys and values, plain query), the others from the
 * INT2 pool (rotated centred keys with the rotated query, values rotated back).
 * All logits are on one scale: the INT2 ones add back q . mu, the constant the
 * key centring removed ("What carries the argument", mechanism 2).
 *   bf16_pool / bf16_page_table: the BF16 cache ([batch][max_pages] table).
 *   mu : fp32 [Hkv][D].  out_rotated: output times R_V (the rotated basis). */
int kvqo_decode_window_head(const uint8_t* pool, int num_pool_pages, const uint8_t* bf16_pool,
                            int bf16_num_pool_pages, const int32_t* bf16_page_table, int H,
                            int Hkv, const uint16_t* q, const int32_t* page_table, int max_pages,
                            int b, int seq_len, int hq, int sink, int recent, const float* R,
                            const float* mu, double sm_scale, int out_rotated, double* out) {
  int G = H / Hkv, kv = hq / G, skipped = 0;
  const float* RK = R + ((size_t)0 * Hkv + kv) * DIM * DIM;
  const float* RV = R + ((size_t)1 * Hkv + kv) * DIM * DIM;
  double qd[DIM], qrot[DIM], qmu = 0.0;
  for (int d = 0; d < DIM; ++d) qd[d] = (double)kvqo_bf16_to_f32(q[d]);
  kvqo_rotate_f64(qd, RK, DIM, qrot);
  for (int d = 0; d < DIM; ++d) qmu += qd[d] * (double)mu[(size_t)kv * DIM + d];
  int n = seq_len > 0 ? seq_len : 1;
  double* logit = (double*)malloc(sizeof(double) * (size_t)n);
  double* vals = (double*)calloc((size_t)n * DIM, sizeof(double));
  char* used = (char*)calloc((size_t)n, 1);
  uint8_t codes[DIM];
  uint16_t s16, z16;
  double mx = -INFINITY;
  for (int p = 0; p < seq_len; ++p) {
    int in_window = (p < sink) || (p >= seq_len - recent);
    double kk[DIM], vv[DIM];
    if (in_window) {
      const uint8_t* rec = record_of((uint8_t*)bf16_pool, BF16_REC, Hkv, bf16_num_pool_pages,
                                     bf16_page_table, max_pages, b, p, kv);
      if (!rec) { ++skipped; continue; }
      for (int d = 0; d < DIM; ++d) {
        int ok = kvqo_bf16_locate(0, p % PAGE, d), ov = kvqo_bf16_locate(1, p % PAGE, d);
        kk[d] = kvqo_bf16_to_f32((uint16_t)(rec[ok] | (rec[ok + 1] << 8)));
        vv[d] = kvqo_bf16_to_f32((uint16_t)(rec[ov] | (rec[ov + 1] << 8)));
      }
      double acc = 0.0;
      for (int d = 0; d < DIM; ++d) acc += qd[d] * kk[d];
      logit[p] = sm_scale * acc;
    } else {
      const uint8_t* rec = record_of((uint8_t*)pool, INT2_REC, Hkv, num_pool_pages, page_table,
                                     max_pages, b, p, kv);
      if (!rec) { ++skipped; continue; }
      kvqo_int2_load(rec, 0, p % PAGE, codes, &s16, &z16);
      double s = kvqo_f16_to_f32(s16), z = kvqo_f16_to_f32(z16);
      double acc = 0.0;
      for (int d = 0; d < DIM; ++d) acc += qrot[d] * ((double)codes[d] * s + z);
      logit[p] = sm_scale * (acc + qmu);
      kvqo_int2_load(rec, 1, p % PAGE, codes, &s16, &z16);
      s = kvqo_f16_to_f32(s16);
      z = kvqo_f16_to_f32(z16);
      double vrot[DIM];
      for (int d = 0; d < DIM; ++d) vrot[d] = (double)codes[d] * s + z;
      kvqo_rotate_t_f64(vrot, RV, DIM, vv);
    }
    for (int d = 0; d < DIM; ++d) vals[(size_t)p * DIM + d] = vv[d];
    used[p] = 1;
    if (logit[p] > mx) mx = logit[p];
  }
  double o[DIM], sum = 0.0;
  for (int d = 0; d < DIM; ++d) o[d] = 0.0;
  for (int p = 0; p < seq_len; ++p) {
    if (!used[p]) continue;
    double w = exp(logit[p] - mx);
    sum += w;
    for (int d = 0; d < DIM; ++d) o[d] += w * vals[(size_t)p * DIM + d];
  }
  for (int d = 0; d < DIM; ++d) o[d] = sum > 0.0 ? o[d] / sum : 0.0;
  if (out_rotated) {
    kvqo_rotate_f64(o, RV, DIM, out);
  } else {
    for (int d = 0; d < DIM; ++d) out[d] = o[d];
  }
  free(logit);
  free(vals);
  free(used);
  return skipped;
}

/* Decode a list of (b, hq) pairs.  pairs : int32 [npairs][2]; out : [npairs][D].
 * q : bf16 [batch][H][D]; seq_lens : [batch].  kind 0 = INT2, 1 = BF16. */
int kvqo_decode_window_pairs(const uint8_t* pool, int num_pool_pages, const uint8_t* bf16_pool,
                             int bf16_num_pool_pages, const int32_t* bf16_page_table, int H, int Hkv,
                             const uint16_t* q, const int32_t* page_table, int max_pages,
                             const int32_t* seq_lens, const int32_t* pairs, int npairs, int sink,
                             int recent, const float* R, const float* mu, double sm_scale,
                             int out_rotated, double* out) {
  int skipped = 0;
  for (int i = 0; i < npairs; ++i) {
    int b = pairs[2 * i], hq = pairs[2 * i + 1];
    skipped += kvqo_decode_window_head(pool, num_pool_pages, bf16_pool, bf16_num_pool_pages,
                                       bf16_page_table, H, Hkv, q + ((size_t)b * H + hq) * DIM,
                                       page_table, max_pages, b, seq_lens[b], hq, sink, recent, R,
                                       mu, sm_scale, out_rotated, out + (size_t)i * DIM);
  }
  return skipped;
}

int kvqo_decode_pairs(int kind, const uint8_t* pool, int num_pool_pages, int H, int Hkv,
                      const uint16_t* q, const int32_t* page_table, int max_pages,
                      const int32_t* seq_lens, const int32_t* pairs, int npairs, const float* R,
                      double sm_scale, int out_rotated, double* out) {
  int skipped = 0;
  for (int i = 0; i < npairs; ++i) {
    int b = pairs[2 * i], hq = pairs[2 * i + 1];
    const uint16_t* qp = q + ((size_t)b * H + hq) * DIM;
    if (kind == 0)
      skipped += kvqo_decode_int2_head(pool, num_pool_pages, H, Hkv, qp, page_table, max_pages, b,
                                       seq_lens[b], hq, R, sm_scale, out_rotated,
                                       out + (size_t)i * DIM);
    else
      skipped += kvqo_decode_bf16_head(pool, num_pool_pages, H, Hkv, qp, page_table, max_pages,
                                       b, seq_lens[b], hq, sm_scale, out + (size_t)i * DIM);
  }
  return skipped;
}
