/*
 * CPU oracle of the Flint NVFP4 W4A16 routed-expert MoE block.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this library.  It shares
 * no code, header, table or helper with the CUDA path; both sides only read
 * the same seeded input bytes.
 *
 * Source of every rule: the vLLM API page "vllm.models.flint.ops.moe"
 * (module docstring, "Numerics"), together with the docstrings of
 * _router_kernel, _topk_row, _gate_up_gemv_kernel, _down_gemv_kernel and
 * _combine_kernel on that page, and the class docstring of
 * vllm.models.flint.model (sigmoid top-k with renormalised weights, ungated
 * shared expert).
 *
 * Plain, slow and sequential: one token at a time, every intermediate held
 * in the type the pages name.  Compile with -O2 -ffp-contract=off and without
 * fast-math so that each C operator is one IEEE-754 operation.
 *
 * Readings taken where the pages are silent:
 *  R1  router-logit summation order (the pages use a Triton tree sum): 32
 *      fp32 partial sums, partial l holding the products of the elements h
 *      with (h / 8) mod 32 == l in ascending h, then combined by the xor
 *      butterfly with offsets 16, 8, 4, 2, 1 as seen from lane 0.
 *  R2  the routing-weight sum over the k selected experts is taken in rank
 *      order.
 *  R3  e2m1 nibble order inside a byte: even K index in the low nibble.
 *  R4  silu(g) = g * sigmoid(g) with an accurately rounded sigmoid; the
 *      product with u is formed last (act = bf16(silu(g) * u)).
 *  R5  the shared expert is a stock BF16 SwiGLU MLP: gS, uS = bf16(fp32 dot),
 *      sact = bf16(silu(gS) * uS) with the stock form silu(v) = v / (1 +
 *      exp(-v)) (accurately rounded exp, fp32 division), ys = bf16(fp32
 *      dot(sact, Wd)).
 *  R6  ranking uses the pages' total order on bf16 bit patterns (numeric
 *      order, except that -0 ranks below +0); equal bit patterns go to the
 *      lower expert index.
 *  R8  add-RMSNorm (_add_rms_norm on the same page, used by flint_moe_ll):
 *      s = a + r in fp32, residual' = bf16(s); the sum of squares, whose
 *      order the page's tree sum leaves open, is the exact sum of the fp32
 *      squares rounded once to fp32 (as R7); v = sum / H + eps in fp32;
 *      the page names the reciprocal square root (_rsqrt) without defining
 *      it: inv = 1 / sqrt(v) correctly rounded to fp32;
 *      xn = bf16((s * inv) * w), each product one fp32 rounding.
 *  R9  BF16 routed experts (flint_moe_bf16_decode on the same page): the
 *      same routing; g, u = fp32(exact dot) of x with BF16 w13 rows (R7),
 *      act = bf16(silu(g) * u) (R4 form), y_e = bf16(fp32(exact dot)) of act
 *      with BF16 w2 rows (no global scale), routed = bf16(sum_j tw_j y_j) in
 *      fp32 rank order, out = bf16(routed + shared_output) with the shared
 *      expert's output given (zero when absent).  The pages store the BF16
 *      experts in a blocked order (BlockMajorK); here they are row-major
 *      [E, 2I, H] and [E, H, I].
 *  R10 an NVFP4 shared expert (LLMoEWeights on the same page: ModelOpt-packed
 *      gate/up and down with block scales and an fp32 global scale each)
 *      follows the routed experts' rule, as the page passes it to the same
 *      kernels: g, u = fp32(exact dot) * gs_gu, sact = bf16(silu(g) * u)
 *      (R4 form), ys = bf16(fp32(exact dot(sact, Wd)) * gs_d); the block's
 *      output is then bf16(bf16(routed) + ys) as with the BF16 shared expert.
 *  R11 fused decode qkv (flint_qkv_fused on the page
 *      "vllm.models.flint.ops.qkv_fused": add-RMSNorm, the qkv GEMV, per-head
 *      q/k RMSNorm, NeoX RoPE and the paged KV-cache write).  xn follows R8
 *      (with no residual: s = x and no residual output); qkv = bf16(fp32(exact
 *      dot(xn, W row)) * gs) for NVFP4 weights (the routed rule, R7), bf16(fp32
 *      exact dot) for BF16 weights; rows [0, nq*128) are the q heads, then
 *      nkv k heads, then nkv v heads.  The NVFP4 scales are taken row-major
 *      [N, H/16] (the MoE experts' order; the page's 128x4-swizzled order is
 *      a permutation of the same bytes).  q/k head norm (qk_norm_rope_cache is
 *      not on the pages; its order of the squares is left open): ss = exact
 *      sum of the squares of the head's 128 bf16 values rounded once to fp32,
 *      v = ss / 128 + qk_eps in fp32, inv = 1 / sqrt(v) correctly rounded,
 *      n = (q * inv) * w in fp32, kept in fp32 for RoPE ("FP32 math"); NeoX
 *      RoPE with c, s = the fp32 table's cos | sin at the token's position:
 *      o[d] = n[d] c[d] - n[d+64] s[d], o[d+64] = n[d+64] c[d] + n[d] s[d]
 *      for d < 64, each product and the sum one fp32 rounding; o = n without
 *      a table; then bf16.  q heads go to q; k heads (o) and v heads (the qkv
 *      values) go to the paged caches at slot = slot_mapping[t] (block
 *      slot / block_size, offset slot % block_size), for t < the mapping's
 *      length and slot >= 0 only.
 *  R7  "products are accumulated in fp32" fixes the accumulator's type, not
 *      the order of the additions.  Every expert and shared-expert dot
 *      product therefore takes the order-independent value: the exact sum of
 *      the (exact) products, rounded once to the fp32 accumulator.  The sum
 *      is formed in double; products of <= 13 significant bits summed over
 *      <= 2^16 terms lose nothing unless the terms span more than ~2^24 in
 *      magnitude, far below fp32 resolution.  The router logits keep the
 *      fixed fp32 order of R1 (ids must be reproducible bit for bit), and the
 *      weighted combine keeps the pages' sequential fp32 loop over j.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- bf16 --- */

/* bf16 -> fp32 is exact: the bf16 pattern is the top half of the fp32 one. */
static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* fp32 -> bf16, round to nearest, ties to even (the rounding every "bf16(.)"
 * on the pages denotes).  NaN stays NaN (quiet bit forced). */
static uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
    return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

static float round_bf16(float f) { return bf16_to_f32(f32_to_bf16(f)); }

/* ------------------------------------------------------ NVFP4 decoding --- */

/* E2M1 (OCP MX FP4): bit 3 sign, bits 2..1 exponent (bias 1), bit 0
 * mantissa.  Exponent 0 is subnormal: value = mantissa * 0.5. */
static float e2m1_value(unsigned code) {
  unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
  float mag = (e == 0) ? 0.5f * (float)m : ldexpf(1.0f + 0.5f * (float)m, (int)e - 1);
  return s ? -mag : mag;
}

/* E4M3 "fn" (float8_e4m3fn): bit 7 sign, bits 6..3 exponent (bias 7), bits
 * 2..0 mantissa.  Exponent 0 is subnormal (m * 2^-9); S.1111.111 is NaN;
 * there is no infinity. */
static float e4m3_value(unsigned byte) {
  unsigned s = (byte >> 7) & 1u, e = (byte >> 3) & 15u, m = byte & 7u;
  float mag;
  if (e == 15 && m == 7)
    return NAN;
  if (e == 0)
    mag = ldexpf((float)m, -9);
  else
    mag = ldexpf(1.0f + (float)m / 8.0f, (int)e - 7);
  return s ? -mag : mag;
}

static float g_e2m1[16];
static float g_e4m3[256];

/* Value tables filled from the two definitions above (speed only). */
static void init_tables(void) {
  for (unsigned c = 0; c < 16; ++c)
    g_e2m1[c] = e2m1_value(c);
  for (unsigned b = 0; b < 256; ++b)
    g_e4m3[b] = e4m3_value(b);
}

/* Dequantised NVFP4 weight element (row-major [rows, K], K/2 bytes per row,
 * one e4m3 scale per 16 consecutive K): e2m1(code) * e4m3(scale), formed in
 * fp32.  The product has at most 5 significant bits, so it is exact. */
static float nvfp4_deq(const uint8_t* codes, const uint8_t* sf, int64_t row, int K, int k) {
  uint8_t byte = codes[row * (K / 2) + k / 2];
  unsigned code = (k & 1) ? (byte >> 4) : (byte & 15u); /* reading R3 */
  return g_e2m1[code] * g_e4m3[sf[row * (K / 16) + k / 16]];
}

/* ------------------------------------------------------------- router --- */

/* bf16 router logit L[t, e] = bf16(sum_h x[t, h] * W[e, h]) with the fp32
 * summation order of reading R1.  Each product of two bf16 values is exact in
 * fp32, so the only roundings are the additions. */
static float router_logit(const uint16_t* xrow, const uint16_t* wrow, int H) {
  float part[32];
  for (int l = 0; l < 32; ++l)
    part[l] = 0.0f;
  for (int h = 0; h < H; ++h) /* ascending h inside every partial */
    part[(h / 8) % 32] = part[(h / 8) % 32] + bf16_to_f32(xrow[h]) * bf16_to_f32(wrow[h]);
  /* xor butterfly: after the step with offset o, lane l holds
   * v[l] + v[l ^ o]; the logit is lane 0's final value. */
  for (int o = 16; o >= 1; o >>= 1) {
    float nxt[32];
    for (int l = 0; l < 32; ++l)
      nxt[l] = part[l] + part[l ^ o];
    memcpy(part, nxt, sizeof(part));
  }
  return round_bf16(part[0]);
}

/* Position of a bf16 bit pattern in the pages' total order (reading R6):
 * non-negative patterns above negative ones, negative ones reversed. */
static unsigned bf16_order(uint16_t b) {
  return (b & 0x8000u) ? (unsigned)(b ^ 0xffffu) : (unsigned)(b | 0x8000u);
}

/* sigmoid in fp32 with an accurately rounded exp: e = fp32(exp(-L)),
 * s = 1 / (1 + e), each step rounded to fp32 (the pages: "exact exp /
 * division"). */
static float sigmoid_exact(float v) {
  float e = (float)exp(-(double)v);
  float d = 1.0f + e;
  return 1.0f / d;
}

/* Top-k of one token's logits, sigmoid scores, renormalised weights rounded
 * to bf16 and stored as fp32, in rank order. */
static void route_token(const uint16_t* logit_bits, int E, int k, int32_t* ids, float* tw) {
  unsigned char taken[256];
  float s[64];
  memset(taken, 0, sizeof(taken));
  for (int j = 0; j < k; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[e])
        continue;
      /* strictly greater keeps the lower index on equal patterns */
      if (best < 0 || bf16_order(logit_bits[e]) > bf16_order(logit_bits[best]))
        best = e;
    }
    taken[best] = 1;
    ids[j] = best;
    s[j] = sigmoid_exact(bf16_to_f32(logit_bits[best]));
  }
  float sum = 0.0f;
  for (int j = 0; j < k; ++j) /* reading R2 */
    sum = sum + s[j];
  float denom = sum + 1e-20f;
  for (int j = 0; j < k; ++j)
    tw[j] = round_bf16(s[j] / denom);
}

/* -------------------------------------------------------------- experts --- */

static float silu_exact(float g) { return g * sigmoid_exact(g); }

/* silu of the stock BF16 SwiGLU layer (reading R5): v / (1 + exp(-v)). */
static float silu_div(float v) {
  float e = (float)exp(-(double)v);
  return v / (1.0f + e);
}

/* One token through the whole block.  Writes out_row[H]; optional
 * intermediates (NULL to skip): ids[k], tw[k], logits[E] (bf16 bits),
 * act[k, I], y[k, H], sact[SI], ys[H] (bf16 bits). */
static void forward_token(const uint16_t* xrow, const uint16_t* wr, const uint8_t* w13,
                          const uint8_t* w13_sf, const float* w13_gs, const uint8_t* w2,
                          const uint8_t* w2_sf, const float* w2_gs, const uint16_t* sgu,
                          const uint16_t* sdown, int H, int E, int k, int I, int SI,
                          uint16_t* out_row, int32_t* ids_o, float* tw_o, uint16_t* logits_o,
                          uint16_t* act_o, uint16_t* y_o, uint16_t* sact_o, uint16_t* ys_o) {
  uint16_t logit_bits[256];
  int32_t ids[64];
  float tw[64];
  float* xf = (float*)malloc(sizeof(float) * (size_t)H);
  float* act = (float*)malloc(sizeof(float) * (size_t)(I > 0 ? I : 1));
  float* R = (float*)calloc((size_t)H, sizeof(float));
  for (int h = 0; h < H; ++h)
    xf[h] = bf16_to_f32(xrow[h]);

  /* router logits and routing */
  for (int e = 0; e < E; ++e)
    logit_bits[e] = f32_to_bf16(router_logit(xrow, wr + (int64_t)e * H, H));
  route_token(logit_bits, E, k, ids, tw);

  /* routed experts, in rank order j = 0 .. k-1 */
  for (int j = 0; j < k; ++j) {
    int64_t e = ids[j];
    const uint8_t* c13 = w13 + e * (int64_t)(2 * I) * (H / 2);
    const uint8_t* s13 = w13_sf + e * (int64_t)(2 * I) * (H / 16);
    float gs13 = w13_gs[e];
    for (int r = 0; r < I; ++r) {
      double sg = 0.0, su = 0.0; /* reading R7 */
      for (int h = 0; h < H; ++h) {
        sg += (double)(nvfp4_deq(c13, s13, r, H, h) * xf[h]);      /* gate row r   */
        su += (double)(nvfp4_deq(c13, s13, I + r, H, h) * xf[h]);  /* up row I + r */
      }
      float accg = (float)sg, accu = (float)su;
      float g = accg * gs13, u = accu * gs13;  /* global scale on the accumulator */
      act[r] = round_bf16(silu_exact(g) * u);  /* act = bf16(silu(g) * u) */
      if (act_o)
        act_o[(int64_t)j * I + r] = f32_to_bf16(act[r]);
    }
    const uint8_t* c2 = w2 + e * (int64_t)H * (I / 2);
    const uint8_t* s2 = w2_sf + e * (int64_t)H * (I / 16);
    float gs2 = w2_gs[e];
    for (int h = 0; h < H; ++h) {
      double sum = 0.0;
      for (int i = 0; i < I; ++i)
        sum += (double)(nvfp4_deq(c2, s2, h, I, i) * act[i]);
      float acc = (float)sum;
      float y = round_bf16(acc * gs2);  /* y_e = bf16(acc * gs_e) */
      if (y_o)
        y_o[(int64_t)j * H + h] = f32_to_bf16(y);
      R[h] = R[h] + tw[j] * y;           /* fp32, sequential in rank j */
    }
  }

  /* shared expert (reading R5) and the final add */
  float* sact = (float*)malloc(sizeof(float) * (size_t)(SI > 0 ? SI : 1));
  for (int r = 0; r < SI; ++r) {
    double sg = 0.0, su = 0.0;
    for (int h = 0; h < H; ++h) {
      sg += (double)(bf16_to_f32(sgu[(int64_t)r * H + h]) * xf[h]);
      su += (double)(bf16_to_f32(sgu[(int64_t)(SI + r) * H + h]) * xf[h]);
    }
    float gS = round_bf16((float)sg), uS = round_bf16((float)su);
    sact[r] = round_bf16(silu_div(gS) * uS);
    if (sact_o)
      sact_o[r] = f32_to_bf16(sact[r]);
  }
  for (int h = 0; h < H; ++h) {
    float ys = 0.0f;
    if (SI > 0) {
      double sum = 0.0;
      for (int i = 0; i < SI; ++i)
        sum += (double)(sact[i] * bf16_to_f32(sdown[(int64_t)h * SI + i]));
      ys = round_bf16((float)sum);
    }
    if (ys_o)
      ys_o[h] = f32_to_bf16(ys);
    out_row[h] = f32_to_bf16(round_bf16(R[h]) + ys);  /* bf16(bf16(routed) + shared) */
  }

  if (ids_o)
    memcpy(ids_o, ids, sizeof(int32_t) * (size_t)k);
  if (tw_o)
    memcpy(tw_o, tw, sizeof(float) * (size_t)k);
  if (logits_o)
    memcpy(logits_o, logit_bits, sizeof(uint16_t) * (size_t)E);
  free(sact);
  free(R);
  free(act);
  free(xf);
}

/* ---------------------------------------------------------------- API --- */

#define ORACLE_API __attribute__((visibility("default")))

static int shape_ok(int M, int H, int E, int k, int I, int SI) {
  return M >= 0 && H > 0 && H % 16 == 0 && E > 0 && E <= 256 && k >= 1 && k <= E &&
         k <= 64 && I >= 0 && I % 16 == 0 && SI >= 0;
}

ORACLE_API float oracle_e2m1_value(int code) { return e2m1_value((unsigned)code & 15u); }
ORACLE_API float oracle_e4m3_value(int byte) { return e4m3_value((unsigned)byte & 255u); }

ORACLE_API void oracle_bf16_round(const float* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i)
    out[i] = f32_to_bf16(in[i]);
}

/* Dequantise a whole NVFP4 matrix [rows, K] to fp32 (pins and diagnostics). */
ORACLE_API void oracle_nvfp4_dequant(const uint8_t* codes, const uint8_t* sf, int64_t rows, int K,
                                     float* out) {
  init_tables();
  for (int64_t r = 0; r < rows; ++r)
    for (int k = 0; k < K; ++k)
      out[r * K + k] = nvfp4_deq(codes, sf, r, K, k);
}

/* Routing only: logits (bf16 bits, optional), ids, tw for all M tokens. */
ORACLE_API int oracle_route(const uint16_t* x, const uint16_t* wr, int M, int H, int E, int k,
                            uint16_t* logits, int32_t* ids, float* tw) {
  if (!shape_ok(M, H, E, k, 0, 0))
    return -1;
  for (int t = 0; t < M; ++t) {
    uint16_t lb[256];
    for (int e = 0; e < E; ++e)
      lb[e] = f32_to_bf16(router_logit(x + (int64_t)t * H, wr + (int64_t)e * H, H));
    if (logits)
      memcpy(logits + (int64_t)t * E, lb, sizeof(uint16_t) * (size_t)E);
    route_token(lb, E, k, ids + (int64_t)t * k, tw + (int64_t)t * k);
  }
  return 0;
}

/* Top-k, sigmoid and renormalisation on given bf16 logits [M, E]. */
ORACLE_API int oracle_topk(const uint16_t* logits, int M, int E, int k, int32_t* ids, float* tw) {
  if (!shape_ok(M, 16, E, k, 0, 0))
    return -1;
  for (int t = 0; t < M; ++t)
    route_token(logits + (int64_t)t * E, E, k, ids + (int64_t)t * k, tw + (int64_t)t * k);
  return 0;
}

/* Whole block for the tokens listed in `tokens` (n_tokens entries; NULL
 * means all M tokens in order).  Row i of every output belongs to
 * tokens[i].  Outputs other than `out` may be NULL.  nthreads <= 0 uses the
 * OpenMP default; tokens are independent, so threads change nothing in the
 * results. */
ORACLE_API int oracle_forward(const uint16_t* x, const uint16_t* wr, const uint8_t* w13,
                              const uint8_t* w13_sf, const float* w13_gs, const uint8_t* w2,
                              const uint8_t* w2_sf, const float* w2_gs, const uint16_t* sgu,
                              const uint16_t* sdown, int M, int H, int E, int k, int I, int SI,
                              const int32_t* tokens, int n_tokens, uint16_t* out, int32_t* ids,
                              float* tw, uint16_t* logits, uint16_t* act, uint16_t* y,
                              uint16_t* sact, uint16_t* ys, int nthreads) {
  if (!shape_ok(M, H, E, k, I, SI))
    return -1;
  init_tables();
  int n = tokens ? n_tokens : M;
  for (int i = 0; i < n; ++i)
    if (tokens && (tokens[i] < 0 || tokens[i] >= M))
      return -1;
#ifdef _OPENMP
  if (nthreads > 0)
    omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int i = 0; i < n; ++i) {
    int64_t t = tokens ? tokens[i] : i;
    forward_token(x + t * H, wr, w13, w13_sf, w13_gs, w2, w2_sf, w2_gs, sgu, sdown, H, E, k, I, SI,
                  out + (int64_t)i * H, ids ? ids + (int64_t)i * k : NULL,
                  tw ? tw + (int64_t)i * k : NULL, logits ? logits + (int64_t)i * E : NULL,
                  act ? act + (int64_t)i * k * I : NULL, y ? y + (int64_t)i * k * H : NULL,
                  sact ? sact + (int64_t)i * SI : NULL, ys ? ys + (int64_t)i * H : NULL);
  }
  return 0;
}

/* NVFP4 shared expert (reading R10) of token rows x [M, H]: ys [M, H] and,
 * optionally, sact [M, SI] (bf16 bits).  sgu codes [2SI, H/2] (gate rows
 * then up rows), sf [2SI, H/16]; sdn codes [H, SI/2], sf [H, SI/16]. */
ORACLE_API int oracle_shared_nvfp4(const uint16_t* x, const uint8_t* sgu, const uint8_t* sgu_sf,
                                   float sgu_gs, const uint8_t* sdn, const uint8_t* sdn_sf,
                                   float sdn_gs, int M, int H, int SI, uint16_t* ys_o,
                                   uint16_t* sact_o) {
  if (M < 0 || H <= 0 || H % 16 != 0 || SI <= 0 || SI % 16 != 0)
    return -1;
  init_tables();
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int t = 0; t < M; ++t) {
    float* xf = (float*)malloc(sizeof(float) * (size_t)H);
    float* sact = (float*)malloc(sizeof(float) * (size_t)SI);
    for (int h = 0; h < H; ++h)
      xf[h] = bf16_to_f32(x[(int64_t)t * H + h]);
    for (int r = 0; r < SI; ++r) {
      double sg = 0.0, su = 0.0; /* reading R7 */
      for (int h = 0; h < H; ++h) {
        sg += (double)(nvfp4_deq(sgu, sgu_sf, r, H, h) * xf[h]);
        su += (double)(nvfp4_deq(sgu, sgu_sf, SI + r, H, h) * xf[h]);
      }
      const float g = (float)sg * sgu_gs, u = (float)su * sgu_gs;
      sact[r] = round_bf16(silu_exact(g) * u);
      if (sact_o)
        sact_o[(int64_t)t * SI + r] = f32_to_bf16(sact[r]);
    }
    for (int h = 0; h < H; ++h) {
      double sum = 0.0;
      for (int i = 0; i < SI; ++i)
        sum += (double)(nvfp4_deq(sdn, sdn_sf, h, SI, i) * sact[i]);
      ys_o[(int64_t)t * H + h] = f32_to_bf16((float)sum * sdn_gs);
    }
    free(xf);
    free(sact);
  }
  return 0;
}

/* BF16 routed experts (reading R9), token rows x [M, H]: out and, optionally,
 * ids / tw [M, k], act [M, k, I] and y [M, k, H] (bf16 bits). */
ORACLE_API int oracle_forward_bf16(const uint16_t* x, const uint16_t* wr, const uint16_t* w13,
                                   const uint16_t* w2, const uint16_t* shared_out, int M, int H,
                                   int E, int k, int I, uint16_t* out, int32_t* ids_o, float* tw_o,
                                   uint16_t* act_o, uint16_t* y_o, int nthreads) {
  if (!shape_ok(M, H, E, k, I, 0))
    return -1;
#ifdef _OPENMP
  if (nthreads > 0)
    omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int t = 0; t < M; ++t) {
    const uint16_t* xrow = x + (int64_t)t * H;
    uint16_t logit_bits[256];
    int32_t ids[64];
    float tw[64];
    float* xf = (float*)malloc(sizeof(float) * (size_t)H);
    float* act = (float*)malloc(sizeof(float) * (size_t)I);
    float* R = (float*)calloc((size_t)H, sizeof(float));
    for (int h = 0; h < H; ++h)
      xf[h] = bf16_to_f32(xrow[h]);
    for (int e = 0; e < E; ++e)
      logit_bits[e] = f32_to_bf16(router_logit(xrow, wr + (int64_t)e * H, H));
    route_token(logit_bits, E, k, ids, tw);
    for (int j = 0; j < k; ++j) {
      const int64_t e = ids[j];
      const uint16_t* g13 = w13 + e * (int64_t)(2 * I) * H;
      for (int r = 0; r < I; ++r) {
        double sg = 0.0, su = 0.0; /* reading R7: bf16 x bf16 products are exact */
        for (int h = 0; h < H; ++h) {
          sg += (double)(bf16_to_f32(g13[(int64_t)r * H + h]) * xf[h]);
          su += (double)(bf16_to_f32(g13[(int64_t)(I + r) * H + h]) * xf[h]);
        }
        const float g = (float)sg, u = (float)su;
        act[r] = round_bf16(silu_exact(g) * u);
        if (act_o)
          act_o[((int64_t)t * k + j) * I + r] = f32_to_bf16(act[r]);
      }
      const uint16_t* g2 = w2 + e * (int64_t)H * I;
      for (int h = 0; h < H; ++h) {
        double sum = 0.0;
        for (int i = 0; i < I; ++i)
          sum += (double)(bf16_to_f32(g2[(int64_t)h * I + i]) * act[i]);
        const float y = round_bf16((float)sum); /* y_e = bf16(acc) */
        if (y_o)
          y_o[((int64_t)t * k + j) * H + h] = f32_to_bf16(y);
        R[h] = R[h] + tw[j] * y;
      }
    }
    for (int h = 0; h < H; ++h) {
      const float sh = shared_out ? bf16_to_f32(shared_out[(int64_t)t * H + h]) : 0.0f;
      out[(int64_t)t * H + h] = f32_to_bf16(round_bf16(R[h]) + sh);
    }
    for (int j = 0; j < k; ++j) {
      if (ids_o)
        ids_o[(int64_t)t * k + j] = ids[j];
      if (tw_o)
        tw_o[(int64_t)t * k + j] = tw[j];
    }
    free(xf);
    free(act);
    free(R);
  }
  return 0;
}

/* norm.fused_add_rms_norm of rows a + r (reading R8): residual' and the
 * normalised rows xn, both bf16 [M, H]; w is the bf16 norm weight [H]. */
ORACLE_API int oracle_add_rms_norm(const uint16_t* a, const uint16_t* r, const uint16_t* w, int M,
                                   int H, float eps, uint16_t* res_out, uint16_t* xn_out) {
  if (M < 0 || H < 1)
    return -1;
  float* s = (float*)malloc(sizeof(float) * (size_t)H);
  if (!s)
    return -1;
  for (int t = 0; t < M; ++t) {
    const uint16_t* at = a + (int64_t)t * H;
    const uint16_t* rt = r + (int64_t)t * H;
    double sq = 0.0; /* squares of fp32 values are exact in double */
    for (int h = 0; h < H; ++h) {
      s[h] = bf16_to_f32(at[h]) + bf16_to_f32(rt[h]);
      res_out[(int64_t)t * H + h] = f32_to_bf16(s[h]);
      sq += (double)s[h] * (double)s[h];
    }
    const float v = (float)sq / (float)H + eps;
    const float inv = (float)(1.0 / sqrt((double)v));
    for (int h = 0; h < H; ++h) {
      const float p = s[h] * inv;
      xn_out[(int64_t)t * H + h] = f32_to_bf16(p * bf16_to_f32(w[h]));
    }
  }
  free(s);
  return 0;
}

/* Fused decode qkv (reading R11) for M tokens: q [M, nq*128] and the cache
 * writes; optionally residual' [M, H] (only with a residual), xn [M, H] and
 * qkv [M, N] (bf16 bits).  Weights: NVFP4 codes [N, H/2] with scales
 * [N, H/16] and global scale gs, or (w_codes NULL) BF16 [N, H].  Caches: bf16
 * element offsets block * s0 + offset * s1 + head * s2 + d. */
ORACLE_API int oracle_qkv_fused(const uint16_t* x, const uint16_t* residual, const uint16_t* norm_w,
                                float eps, const uint8_t* w_codes, const uint8_t* w_sf, float gs,
                                const uint16_t* w_bf16, const uint16_t* q_norm_w,
                                const uint16_t* k_norm_w, float qk_eps, const float* cos_sin,
                                const int64_t* positions, const int64_t* slot_mapping, int n_slots,
                                int M, int H, int nq, int nkv, int block_size, int64_t s0, int64_t s1,
                                int64_t s2, uint16_t* k_cache, uint16_t* v_cache, uint16_t* q_out,
                                uint16_t* res_out, uint16_t* xn_out, uint16_t* qkv_out) {
  enum { D = 128 };
  if (M < 0 || H <= 0 || H % 16 != 0 || nq < 1 || nkv < 0 || block_size < 1)
    return -1;
  if (!w_codes && !w_bf16)
    return -1;
  init_tables();
  const int N = (nq + 2 * nkv) * D;
  float* s = (float*)malloc(sizeof(float) * (size_t)H);
  float* xn = (float*)malloc(sizeof(float) * (size_t)H);
  uint16_t* qkv = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)N);
  if (!s || !xn || !qkv) {
    free(s);
    free(xn);
    free(qkv);
    return -1;
  }
  for (int t = 0; t < M; ++t) {
    /* the input RMSNorm (reading R8) */
    double sq = 0.0;
    for (int h = 0; h < H; ++h) {
      s[h] = bf16_to_f32(x[(int64_t)t * H + h]);
      if (residual) {
        s[h] = s[h] + bf16_to_f32(residual[(int64_t)t * H + h]);
        if (res_out)
          res_out[(int64_t)t * H + h] = f32_to_bf16(s[h]);
      }
      sq += (double)s[h] * (double)s[h];
    }
    const float v = (float)sq / (float)H + eps;
    const float inv = (float)(1.0 / sqrt((double)v));
    for (int h = 0; h < H; ++h) {
      xn[h] = round_bf16((s[h] * inv) * bf16_to_f32(norm_w[h]));
      if (xn_out)
        xn_out[(int64_t)t * H + h] = f32_to_bf16(xn[h]);
    }
    /* the qkv GEMV (reading R7 sums) */
    for (int n = 0; n < N; ++n) {
      double acc = 0.0;
      if (w_codes) {
        for (int h = 0; h < H; ++h)
          acc += (double)(nvfp4_deq(w_codes, w_sf, n, H, h) * xn[h]);
        qkv[n] = f32_to_bf16((float)acc * gs);
      } else {
        for (int h = 0; h < H; ++h)
          acc += (double)(bf16_to_f32(w_bf16[(int64_t)n * H + h]) * xn[h]);
        qkv[n] = f32_to_bf16((float)acc);
      }
      if (qkv_out)
        qkv_out[(int64_t)t * N + n] = qkv[n];
    }
    const int64_t slot = t < n_slots ? slot_mapping[t] : -1;
    const int64_t cache_row = slot >= 0 ? (slot / block_size) * s0 + (slot % block_size) * s1 : 0;
    /* q and k heads: norm, RoPE */
    for (int hh = 0; hh < nq + nkv; ++hh) {
      const uint16_t* hv = qkv + hh * D;
      const uint16_t* nw = hh < nq ? q_norm_w : k_norm_w;
      double hs = 0.0;
      for (int d = 0; d < D; ++d)
        hs += (double)bf16_to_f32(hv[d]) * (double)bf16_to_f32(hv[d]);
      const float hvar = (float)hs / (float)D + qk_eps;
      const float hinv = (float)(1.0 / sqrt((double)hvar));
      float nrm[D], o[D];
      for (int d = 0; d < D; ++d)
        nrm[d] = (bf16_to_f32(hv[d]) * hinv) * bf16_to_f32(nw[d]);
      if (cos_sin) {
        const float* cs = cos_sin + positions[t] * D;
        for (int d = 0; d < D / 2; ++d) {
          const float c = cs[d], sn = cs[D / 2 + d];
          o[d] = nrm[d] * c - nrm[d + D / 2] * sn;
          o[d + D / 2] = nrm[d + D / 2] * c + nrm[d] * sn;
        }
      } else {
        for (int d = 0; d < D; ++d)
          o[d] = nrm[d];
      }
      for (int d = 0; d < D; ++d) {
        if (hh < nq)
          q_out[(int64_t)t * nq * D + hh * D + d] = f32_to_bf16(o[d]);
        else if (slot >= 0)
          k_cache[cache_row + (int64_t)(hh - nq) * s2 + d] = f32_to_bf16(o[d]);
      }
    }
    /* v heads: the qkv values */
    for (int vh = 0; vh < nkv && slot >= 0; ++vh)
      for (int d = 0; d < D; ++d)
        v_cache[cache_row + (int64_t)vh * s2 + d] = qkv[(nq + nkv + vh) * D + d];
  }
  free(s);
  free(xn);
  free(qkv);
  return 0;
}

ORACLE_API int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
