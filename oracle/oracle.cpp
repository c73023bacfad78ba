/*
 * oracle.cpp -- plain, slow CPU restatement of the Qwen2-style prefill
 * forward with Q8_0 weights and on-the-fly Q8_0 activations.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the bench's CPU
 * baseline do.  It shares no code with the CUDA path.
 *
 * Sources (minfer "Inference E2E Walkthrough" pages):
 *   [P09]   "09 · Prefill: the first forward"
 *   [INDEX] "minfer Inference E2E Walkthrough — one run, stage by stage"
 *           (master table, rows "CPU matmul kernels" and
 *           "Attention + vec ops + KV")
 *   [P05]   "05 · Graph build — the IR and the builder"
 *
 * Readings taken where the pages are silent (each is listed with its reason
 * in the design notes):
 *   R1 Q8_0 block = 32 int8 codes + one fp16 scale; d = amax/127 in f32,
 *      codes = roundf(x * (1/d)) (ties away from zero), scale stored as the
 *      round-to-nearest-even fp16 of d.  A row whose length is not a multiple
 *      of 32 ends in a partial block whose missing elements count as zero.
 *   R2 Matmul: per 32-block int32 dot, each scaled by f32(dw)*f32(da), summed
 *      over blocks in double, rounded to f32, then the bias added in f32.
 *   R3 RMSNorm: mean of squares accumulated in double; eps added in double;
 *      scale rounded to f32; y = (x * scale) * w in f32.
 *   R4 RoPE: NeoX half-split pairs (i, i + hd/2), angle pos * theta^(-2i/hd)
 *      in double, cos/sin rounded to f32.
 *   R5 Attention: query head h reads KV head h / (n_head / n_head_kv);
 *      scores and softmax in double; KV rows never written read as zero.
 *   R6 SiLU(g) * u evaluated in double, rounded to f32.
 *   R7 argmax ties go to the lowest index.
 *   R8 Qwen3 QK-norm ([P05] section 2.5 operation family "qk_norm (Qwen3)";
 *      section 3.2 "FusedQkvNorm": the per-head Q/K RMSNorm sits between the
 *      three matmuls and the two RoPEs): each head of Q and of K is RMS-
 *      normalized over its head_dim values as in R3, with one weight vector
 *      of head_dim entries per layer for Q and one for K, after the bias and
 *      before RoPE.  Models with QK-norm carry no Q/K/V bias.
 *   R9 Positions within one call are distinct; a repeated position is
 *      rejected as a bad argument before anything is written.
 *
 * Every floating-point statement below is evaluated exactly as written: the
 * file is compiled with -ffp-contract=off and without fast-math.
 *
 * Parity status per function (what pins it, checked by the CPU tests):
 *   q8 codec        -- brute force over all codes, scale/2 bound, specials
 *   block dots      -- brute-force integer sums
 *   matmul          -- dequantize-then-float64-GEMM closed form (numpy)
 *   rmsnorm         -- float64 closed form (numpy), scale invariance
 *   qk-norm         -- per-head rmsnorm; in the model: logits invariant to a
 *                      power-of-two scaling of Wq/Wk (and not without it)
 *   rope            -- norm preservation, R(a)R(b)=R(a+b), relative-position
 *                      property, a single-unit-vector closed form
 *   attention       -- brute-force masked softmax(QK^T/sqrt(d))V (numpy)
 *   swiglu          -- float64 closed form (numpy)
 *   argmax          -- brute force over vectors with planted ties
 *   model prefill   -- invariants only: causality, one-shot == token by
 *                      token, n_out=1 == last row of n_out=nt, written-slot
 *                      set, zero-weight special case.  The composition itself
 *                      has no printed values on the pages: parity unpinned
 *                      beyond those invariants.
 */
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <map>
#include <string>
#include <vector>

namespace {

/* ---------- IEEE 754 binary16 conversions (from the format definition) ---------- */

uint32_t f32_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return u;
}

/* f32 -> binary16, round to nearest, ties to even. */
uint16_t f32_to_f16(float f) {
  const uint32_t x = f32_bits(f);
  const uint32_t sign = (x >> 16) & 0x8000u;
  const uint32_t ax = x & 0x7FFFFFFFu;
  if (ax >= 0x7F800000u) return (uint16_t)(sign | 0x7C00u | (ax > 0x7F800000u ? 0x200u : 0u));
  if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u); /* >= 65520 rounds to inf */
  if (ax <= 0x33000000u) return (uint16_t)sign;              /* <= 2^-25 rounds to 0 */
  const int e = (int)(ax >> 23) - 127;
  const uint32_t m = (ax & 0x7FFFFFu) | 0x800000u; /* 24-bit significand */
  if (e < -14) {
    /* subnormal: value = m * 2^(e-23) = code * 2^-24 -> code = m >> (-(e+1)) */
    const int s = -(e + 1);
    uint32_t q = m >> s;
    const uint32_t rem = m & ((1u << s) - 1u);
    const uint32_t half = 1u << (s - 1);
    if (rem > half || (rem == half && (q & 1u))) ++q;
    return (uint16_t)(sign | q);
  }
  uint32_t q = (ax & 0x7FFFFFu) >> 13;
  const uint32_t rem = ax & 0x1FFFu;
  uint32_t r = ((uint32_t)(e + 15) << 10) + q;
  if (rem > 0x1000u || (rem == 0x1000u && (q & 1u))) ++r;
  return (uint16_t)(sign | r);
}

float f16_to_f32(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int ex = (h >> 10) & 0x1F;
  const int mant = h & 0x3FF;
  double v;
  if (ex == 0) v = std::ldexp((double)mant, -24);
  else if (ex == 31) v = mant ? NAN : INFINITY;
  else v = std::ldexp(1024.0 + mant, ex - 25);
  return (float)(sign ? -v : v);
}

/* ---------- Q8_0 (reading R1; [INDEX] row "CPU matmul kernels": quantized
 * weight x on-the-fly Q8_0 activations) ---------- */

void quantize_row(const float* x, int64_t n, int8_t* q, uint16_t* d) {
  const int64_t nb = (n + 31) / 32;
  for (int64_t b = 0; b < nb; ++b) {
    const int64_t k0 = 32 * b, k1 = std::min<int64_t>(n, k0 + 32);
    float amax = 0.0f;
    for (int64_t k = k0; k < k1; ++k) amax = std::max(amax, std::fabs(x[k]));
    const float dd = amax / 127.0f;
    const float id = dd != 0.0f ? 1.0f / dd : 0.0f;
    for (int64_t k = k0; k < k0 + 32; ++k) {
      if (k >= k1) { q[k] = 0; continue; }
      float r = std::round(x[k] * id);
      r = std::min(127.0f, std::max(-127.0f, r));
      q[k] = (int8_t)r;
    }
    d[b] = f32_to_f16(dd);
  }
}

/* A Q8_0 matrix: rows x (nb*32) codes (zero padded), rows x nb scales. */
struct QMat {
  int64_t rows = 0, cols = 0, nb = 0;
  std::vector<int8_t> q;
  std::vector<uint16_t> d;
  bool present = false;
};

void qmat_from_f32(QMat& m, const float* x, int64_t rows, int64_t cols) {
  m.rows = rows; m.cols = cols; m.nb = (cols + 31) / 32;
  m.q.assign(rows * m.nb * 32, 0);
  m.d.assign(rows * m.nb, 0);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    quantize_row(x + r * cols, cols, m.q.data() + r * m.nb * 32, m.d.data() + r * m.nb);
  m.present = true;
}

/* 34-byte blocks: uint16 scale bits (little endian), 32 int8 codes. */
void qmat_from_blocks(QMat& m, const uint8_t* blk, int64_t rows, int64_t cols) {
  m.rows = rows; m.cols = cols; m.nb = (cols + 31) / 32;
  m.q.assign(rows * m.nb * 32, 0);
  m.d.assign(rows * m.nb, 0);
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < m.nb; ++b) {
      const uint8_t* p = blk + 34 * (r * m.nb + b);
      m.d[r * m.nb + b] = (uint16_t)(p[0] | (p[1] << 8));
      for (int k = 0; k < 32; ++k) {
        const int64_t c = 32 * b + k;
        m.q[(r * m.nb + b) * 32 + k] = c < cols ? (int8_t)p[2 + k] : 0;
      }
    }
  m.present = true;
}

/* Quantized matmul (reading R2).  x: Q8_0 rows [M][nb*32] + scales [M][nb];
 * W: Q8_0 [N][nb*32]; y[m][n] = f32(sum_b dw*da*isum_b) (+ bias[n]).
 * [P05] section 3.2 "The builder in practice": the bias rides along with the
 * matmul and is applied inline. */
void matmul_q8(const int8_t* xq, const uint16_t* xd, int64_t M, const QMat& w,
               const float* bias, float* y) {
  const int64_t nb = w.nb, N = w.rows;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t m = 0; m < M; ++m) {
    const int8_t* a = xq + m * nb * 32;
    const uint16_t* da = xd + m * nb;
    for (int64_t n = 0; n < N; ++n) {
      const int8_t* b = w.q.data() + n * nb * 32;
      const uint16_t* dw = w.d.data() + n * nb;
      double acc = 0.0;
      for (int64_t k = 0; k < nb; ++k) {
        int32_t s = 0;
        for (int i = 0; i < 32; ++i) s += (int32_t)a[32 * k + i] * (int32_t)b[32 * k + i];
        acc += (double)f16_to_f32(dw[k]) * (double)f16_to_f32(da[k]) * (double)s;
      }
      float v = (float)acc;
      if (bias) v = v + bias[n];
      y[m * N + n] = v;
    }
  }
}

/* RMSNorm (reading R3; [P05] section 2.5 node list: rms_norm "attn_norm",
 * "ffn_norm", final norm, eps 1e-6). */
void rmsnorm_row(const float* x, const float* w, int64_t n, float eps, float* y) {
  double ss = 0.0;
  for (int64_t i = 0; i < n; ++i) ss += (double)x[i] * (double)x[i];
  const float r = (float)(1.0 / std::sqrt(ss / (double)n + (double)eps));
  for (int64_t i = 0; i < n; ++i) {
    const float t = x[i] * r;
    y[i] = t * w[i];
  }
}

/* RoPE tables (reading R4): cos/sin of pos * theta^(-2i/hd), [n_ctx][hd/2]. */
void rope_table(int n_ctx, int hd, float theta, float* c, float* s) {
  const int half = hd / 2;
  for (int i = 0; i < half; ++i) {
    const double inv_freq = std::pow((double)theta, -2.0 * (double)i / (double)hd);
    for (int p = 0; p < n_ctx; ++p) {
      const double a = (double)p * inv_freq;
      c[(int64_t)p * half + i] = (float)std::cos(a);
      s[(int64_t)p * half + i] = (float)std::sin(a);
    }
  }
}

/* Rotate every head of x[t] ([nt][nheads*hd]) by its position ([P09]
 * section 2.2: the rope nodes read the positions buffer as the angle input). */
void rope_apply(float* x, int64_t nt, int nheads, int hd, const int32_t* pos,
                const float* c, const float* s) {
  const int half = hd / 2;
  for (int64_t t = 0; t < nt; ++t)
    for (int h = 0; h < nheads; ++h) {
      float* v = x + t * (int64_t)nheads * hd + (int64_t)h * hd;
      const float* cp = c + (int64_t)pos[t] * half;
      const float* sp = s + (int64_t)pos[t] * half;
      for (int i = 0; i < half; ++i) {
        const float a = v[i], b = v[i + half];
        const float ac = a * cp[i], bs = b * sp[i], as = a * sp[i], bc = b * cp[i];
        v[i] = ac - bs;
        v[i + half] = as + bc;
      }
    }
}

/* Rounding variant of the attention, used only to measure how far two
 * correct roundings of the same forward drift apart: 0 = float64 scores,
 * softmax and weighted sum (the reference behaviour), 1 = the same steps in
 * float32. */
int g_attn_f32 = 0;

/* Causal GQA attention (reading R5; [P09] section 2.2: token t attends to
 * positions 0..=pos[t]; [P05] section 2.5: scale 1/sqrt(head_dim), n_head_kv
 * groups).  q: [nt][nh*hd]; K,V regions: [n_ctx][nkv*hd]; o: [nt][nh*hd]. */
void attention(const float* q, int64_t nt, const int32_t* pos, const float* K, const float* V,
               int nh, int nkv, int hd, float* o) {
  const int group = nh / nkv;
  const int64_t kvw = (int64_t)nkv * hd;
  const double scale = 1.0 / std::sqrt((double)hd);
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
  for (int64_t t = 0; t < nt; ++t)
    for (int h = 0; h < nh; ++h) {
      const int g = h / group;
      const float* qv = q + t * (int64_t)nh * hd + (int64_t)h * hd;
      const int64_t nk = (int64_t)pos[t] + 1;
      if (g_attn_f32) {
        std::vector<float> sf(nk);
        float mf = -INFINITY;
        const float fscale = 1.0f / std::sqrt((float)hd);
        for (int64_t j = 0; j < nk; ++j) {
          const float* kr = K + j * kvw + (int64_t)g * hd;
          float dot = 0.0f;
          for (int d = 0; d < hd; ++d) dot = dot + qv[d] * kr[d];
          sf[j] = dot * fscale;
          mf = std::max(mf, sf[j]);
        }
        float denf = 0.0f;
        for (int64_t j = 0; j < nk; ++j) { sf[j] = std::exp(sf[j] - mf); denf = denf + sf[j]; }
        float* ovf = o + t * (int64_t)nh * hd + (int64_t)h * hd;
        for (int d = 0; d < hd; ++d) {
          float acc = 0.0f;
          for (int64_t j = 0; j < nk; ++j) acc = acc + sf[j] * V[j * kvw + (int64_t)g * hd + d];
          ovf[d] = acc / denf;
        }
        continue;
      }
      std::vector<double> sc(nk);
      double mx = -INFINITY;
      for (int64_t j = 0; j < nk; ++j) {
        const float* kr = K + j * kvw + (int64_t)g * hd;
        double dot = 0.0;
        for (int d = 0; d < hd; ++d) dot += (double)qv[d] * (double)kr[d];
        sc[j] = dot * scale;
        mx = std::max(mx, sc[j]);
      }
      double den = 0.0;
      for (int64_t j = 0; j < nk; ++j) { sc[j] = std::exp(sc[j] - mx); den += sc[j]; }
      float* ov = o + t * (int64_t)nh * hd + (int64_t)h * hd;
      for (int d = 0; d < hd; ++d) {
        double acc = 0.0;
        for (int64_t j = 0; j < nk; ++j) acc += sc[j] * (double)V[j * kvw + (int64_t)g * hd + d];
        ov[d] = (float)(acc / den);
      }
    }
}

/* SwiGLU (reading R6; [P05] section 2.5: silu(gate) * up). */
float swiglu(float g, float u) {
  const double gd = (double)g;
  return (float)(gd / (1.0 + std::exp(-gd)) * (double)u);
}

}  // namespace

/* ============================== C ABI ============================== */

extern "C" {

typedef struct {
  int n_layer, n_embd, n_head, n_head_kv, head_dim, n_ff, n_vocab, max_seq_len;
  float rope_theta, rms_eps;
  int tied_embeddings;
  int qk_norm; /* reading R8 */
} orc_hparams;

struct OrcLayer {
  std::vector<float> attn_norm, ffn_norm, bq, bk, bv, q_norm, k_norm;
  QMat wq, wk, wv, wo, wg, wu, wd;
};

struct orc_model {
  orc_hparams hp;
  QMat tok_embd, output;
  std::vector<float> out_norm;
  std::vector<OrcLayer> layers;
};

struct orc_kv {
  int n_ctx = 0;
  std::vector<std::vector<float>> k, v; /* per layer [n_ctx][nkv*hd] */
};

uint16_t orc_f32_to_f16(float f) { return f32_to_f16(f); }

/* Select the attention rounding variant (see g_attn_f32); returns the old one. */
int orc_set_attention_f32(int on) {
  const int old = g_attn_f32;
  g_attn_f32 = on ? 1 : 0;
  return old;
}
float orc_f16_to_f32(uint16_t h) { return f16_to_f32(h); }

/* Quantize rows x [rows][n] -> codes [rows][nb*32], scale bits [rows][nb]. */
void orc_q8_quantize(const float* x, int64_t rows, int64_t n, int8_t* q, uint16_t* d) {
  const int64_t nb = (n + 31) / 32;
  for (int64_t r = 0; r < rows; ++r) quantize_row(x + r * n, n, q + r * nb * 32, d + r * nb);
}

void orc_q8_dequantize(const int8_t* q, const uint16_t* d, int64_t rows, int64_t n, float* x) {
  const int64_t nb = (n + 31) / 32;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t k = 0; k < n; ++k)
      x[r * n + k] = f16_to_f32(d[r * nb + k / 32]) * (float)q[r * nb * 32 + k];
}

/* Per-32-block int32 dots: out[m][n][b] = sum_i qa[m][32b+i] * qw[n][32b+i]. */
void orc_block_dots(const int8_t* qa, int64_t M, const int8_t* qw, int64_t N, int64_t nb,
                    int32_t* out) {
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n)
      for (int64_t b = 0; b < nb; ++b) {
        int32_t s = 0;
        for (int i = 0; i < 32; ++i)
          s += (int32_t)qa[(m * nb + b) * 32 + i] * (int32_t)qw[(n * nb + b) * 32 + i];
        out[(m * N + n) * nb + b] = s;
      }
}

/* y[M][N] = Q8_0(x) . Q8_0(W)^T (+ bias).  Operands already quantized. */
void orc_matmul_q8(const int8_t* xq, const uint16_t* xd, int64_t M, const int8_t* wq,
                   const uint16_t* wd, int64_t N, int64_t K, const float* bias, float* y) {
  QMat w;
  w.rows = N; w.cols = K; w.nb = (K + 31) / 32;
  w.q.assign(wq, wq + N * w.nb * 32);
  w.d.assign(wd, wd + N * w.nb);
  matmul_q8(xq, xd, M, w, bias, y);
}

void orc_rmsnorm(const float* x, const float* w, int64_t rows, int64_t n, float eps, float* y) {
  for (int64_t r = 0; r < rows; ++r) rmsnorm_row(x + r * n, w, n, eps, y + r * n);
}

void orc_rope_table(int n_ctx, int hd, float theta, float* c, float* s) {
  rope_table(n_ctx, hd, theta, c, s);
}

void orc_rope(float* x, int64_t nt, int nheads, int hd, const int32_t* pos, const float* c,
              const float* s) {
  rope_apply(x, nt, nheads, hd, pos, c, s);
}

void orc_attention(const float* q, int64_t nt, const int32_t* pos, const float* K,
                   const float* V, int nh, int nkv, int hd, float* o) {
  attention(q, nt, pos, K, V, nh, nkv, hd, o);
}

void orc_swiglu(const float* g, const float* u, int64_t n, float* s) {
  for (int64_t i = 0; i < n; ++i) s[i] = swiglu(g[i], u[i]);
}

/* ---------------- model ---------------- */

orc_model* orc_model_create(const orc_hparams* hp) {
  if (!hp || hp->n_layer <= 0 || hp->n_head <= 0 || hp->n_head_kv <= 0 ||
      hp->n_head % hp->n_head_kv != 0 || hp->head_dim % 2 != 0)
    return nullptr;
  orc_model* m = new orc_model();
  m->hp = *hp;
  m->layers.resize(hp->n_layer);
  return m;
}

void orc_model_free(orc_model* m) { delete m; }

static bool parse_layer(const char* name, int* layer, std::string* kind) {
  if (std::strncmp(name, "blk.", 4) != 0) return false;
  char* end = nullptr;
  const long l = std::strtol(name + 4, &end, 10);
  if (!end || *end != '.') return false;
  *layer = (int)l;
  *kind = std::string(end + 1);
  return true;
}

/* Locate a tensor slot by GGUF name.  Returns 0 and fills exactly one of
 * *qm / *vec, or -1 for an unknown name or layer. */
static int lookup(orc_model* m, const char* name, QMat** qm, std::vector<float>** vec,
                  int64_t* ne0, int64_t* ne1) {
  const orc_hparams& hp = m->hp;
  const int64_t H = hp.n_embd, q = (int64_t)hp.n_head * hp.head_dim,
                kv = (int64_t)hp.n_head_kv * hp.head_dim, F = hp.n_ff, V = hp.n_vocab;
  *qm = nullptr; *vec = nullptr;
  const std::string s(name);
  if (s == "token_embd.weight") { *qm = &m->tok_embd; *ne0 = H; *ne1 = V; return 0; }
  if (s == "output.weight") { *qm = &m->output; *ne0 = H; *ne1 = V; return 0; }
  if (s == "output_norm.weight") { *vec = &m->out_norm; *ne0 = H; *ne1 = 1; return 0; }
  int l;
  std::string k;
  if (!parse_layer(name, &l, &k) || l < 0 || l >= hp.n_layer) return -1;
  OrcLayer& L = m->layers[l];
  if (k == "attn_norm.weight") { *vec = &L.attn_norm; *ne0 = H; *ne1 = 1; return 0; }
  if (k == "ffn_norm.weight") { *vec = &L.ffn_norm; *ne0 = H; *ne1 = 1; return 0; }
  if (k == "attn_q.bias") { *vec = &L.bq; *ne0 = q; *ne1 = 1; return 0; }
  if (k == "attn_k.bias") { *vec = &L.bk; *ne0 = kv; *ne1 = 1; return 0; }
  if (k == "attn_v.bias") { *vec = &L.bv; *ne0 = kv; *ne1 = 1; return 0; }
  if (hp.qk_norm && k == "attn_q_norm.weight") { *vec = &L.q_norm; *ne0 = hp.head_dim; *ne1 = 1; return 0; }
  if (hp.qk_norm && k == "attn_k_norm.weight") { *vec = &L.k_norm; *ne0 = hp.head_dim; *ne1 = 1; return 0; }
  if (k == "attn_q.weight") { *qm = &L.wq; *ne0 = H; *ne1 = q; return 0; }
  if (k == "attn_k.weight") { *qm = &L.wk; *ne0 = H; *ne1 = kv; return 0; }
  if (k == "attn_v.weight") { *qm = &L.wv; *ne0 = H; *ne1 = kv; return 0; }
  if (k == "attn_output.weight") { *qm = &L.wo; *ne0 = q; *ne1 = H; return 0; }
  if (k == "ffn_gate.weight") { *qm = &L.wg; *ne0 = H; *ne1 = F; return 0; }
  if (k == "ffn_up.weight") { *qm = &L.wu; *ne0 = H; *ne1 = F; return 0; }
  if (k == "ffn_down.weight") { *qm = &L.wd; *ne0 = F; *ne1 = H; return 0; }
  return -1;
}

/* Set a tensor from f32 data (matrices are quantized to Q8_0 here). */
int orc_model_set_f32(orc_model* m, const char* name, const float* data, int64_t ne0,
                      int64_t ne1) {
  QMat* qm; std::vector<float>* vec; int64_t e0, e1;
  if (lookup(m, name, &qm, &vec, &e0, &e1) != 0) return -1;
  if (e0 != ne0 || e1 != ne1) return -2;
  if (qm) qmat_from_f32(*qm, data, ne1, ne0);
  else vec->assign(data, data + ne0);
  return 0;
}

/* Set a matrix from raw 34-byte Q8_0 blocks (rows of ceil(ne0/32) blocks). */
int orc_model_set_q8_0(orc_model* m, const char* name, const uint8_t* blocks, int64_t ne0,
                       int64_t ne1) {
  QMat* qm; std::vector<float>* vec; int64_t e0, e1;
  if (lookup(m, name, &qm, &vec, &e0, &e1) != 0) return -1;
  if (!qm || e0 != ne0 || e1 != ne1) return -2;
  qmat_from_blocks(*qm, blocks, ne1, ne0);
  return 0;
}

/* Read back a quantized matrix (codes [ne1][nb*32], scale bits [ne1][nb]). */
int orc_model_get_q8(orc_model* m, const char* name, int8_t* q, uint16_t* d) {
  QMat* qm; std::vector<float>* vec; int64_t e0, e1;
  if (lookup(m, name, &qm, &vec, &e0, &e1) != 0 || !qm || !qm->present) return -1;
  std::memcpy(q, qm->q.data(), qm->q.size());
  std::memcpy(d, qm->d.data(), qm->d.size() * 2);
  return 0;
}

/* 0 when every tensor the forward needs is present, else -1. */
int orc_model_check(orc_model* m) {
  if (!m->tok_embd.present || m->out_norm.empty()) return -1;
  if (!m->hp.tied_embeddings && !m->output.present) return -1;
  for (auto& L : m->layers) {
    if (L.attn_norm.empty() || L.ffn_norm.empty() || !L.wq.present || !L.wk.present ||
        !L.wv.present || !L.wo.present || !L.wg.present || !L.wu.present || !L.wd.present)
      return -1;
    /* Qwen2: Q/K/V biases; Qwen3 (R8): the two QK-norm weights, biases optional */
    if (!m->hp.qk_norm && (L.bq.empty() || L.bk.empty() || L.bv.empty())) return -1;
    if (m->hp.qk_norm && (L.q_norm.empty() || L.k_norm.empty())) return -1;
  }
  return 0;
}

/* KV regions ([P09] section 2.5: per layer, K and V regions of
 * n_kv_embd x n_ctx f32, sized once; n_ctx clamped to max_seq_len).
 * Regions start zero-filled (reading R5). */
orc_kv* orc_kv_create(orc_model* m, int n_ctx) {
  if (n_ctx <= 0) return nullptr;
  orc_kv* kv = new orc_kv();
  kv->n_ctx = std::min(n_ctx, m->hp.max_seq_len);
  const int64_t w = (int64_t)m->hp.n_head_kv * m->hp.head_dim;
  kv->k.assign(m->hp.n_layer, std::vector<float>(kv->n_ctx * w, 0.0f));
  kv->v.assign(m->hp.n_layer, std::vector<float>(kv->n_ctx * w, 0.0f));
  return kv;
}

void orc_kv_free(orc_kv* kv) { delete kv; }

int orc_kv_ctx(const orc_kv* kv) { return kv->n_ctx; }

/* Copy rows [row0, row0+nrows) of layer's K (which=0) or V (which=1). */
int orc_kv_read(const orc_kv* kv, int layer, int which, int row0, int nrows, float* out,
                int64_t width) {
  if (layer < 0 || layer >= (int)kv->k.size() || row0 < 0 || row0 + nrows > kv->n_ctx) return -1;
  const std::vector<float>& r = which ? kv->v[layer] : kv->k[layer];
  std::memcpy(out, r.data() + (int64_t)row0 * width, sizeof(float) * nrows * width);
  return 0;
}

int orc_kv_write(orc_kv* kv, int layer, int which, int row0, int nrows, const float* in,
                 int64_t width) {
  if (layer < 0 || layer >= (int)kv->k.size() || row0 < 0 || row0 + nrows > kv->n_ctx) return -1;
  std::vector<float>& r = which ? kv->v[layer] : kv->k[layer];
  std::memcpy(r.data() + (int64_t)row0 * width, in, sizeof(float) * nrows * width);
  return 0;
}

/*
 * The prefill forward ([P09] sections 2.2-2.4 and 3.2; [P05] section 2.5
 * node list and section 2.8 tail rows).
 *
 *   h = embed(ids)
 *   per layer: x = Q8_0(rmsnorm(h) * attn_norm)
 *              Q,K,V = x.W{q,k,v} + b
 *              (Qwen3, R8: Q, K = per-head rmsnorm(Q, K) * q_norm, k_norm)
 *              rope(Q), rope(K) at pos
 *              K/V regions row pos[t] <- K[t], V[t]    (before attention)
 *              a = attention(Q, regions, pos)          (all rows)
 *              o = Q8_0(a).Wo
 *              last layer with n_out < nt: keep the tail n_out rows of o and h
 *              h = h + o
 *              x = Q8_0(rmsnorm(h) * ffn_norm)
 *              s = Q8_0(silu(x.Wg) * (x.Wu));  h = h + s.Wd
 *   logits = Q8_0(rmsnorm(h) * output_norm) . W_out   (W_out = tok_embd if tied)
 *
 * Returns 0; -1 bad arguments (including a repeated position, R9); -2 a position outside [0, n_ctx) ([P09]
 * section 3.4: positions must stay below n_ctx); -3 a token id outside the
 * vocabulary; -4 missing tensors.  Errors are detected before anything is
 * written.
 *
 * hidden (optional): [n_layer + 1] slots of [nt][H]; slot 0 is the embedding
 * output, slot l+1 the output of layer l (the last layer's slot holds only the
 * tail rows, in the first n_out rows of the slot).
 */
int orc_prefill(orc_model* m, orc_kv* kv, const int32_t* ids, const int32_t* pos, int nt,
                int n_out, float* logits, float* hidden) {
  if (!m || !kv || !ids || !pos || nt <= 0 || n_out <= 0 || n_out > nt || !logits) return -1;
  for (int t = 0; t < nt; ++t)
    if (pos[t] < 0 || pos[t] >= kv->n_ctx) return -2;
  /* reading R9: one call writes each region row at most once ([P09] section
     2.2 gives every token its own slot); a repeated position is a bad argument */
  {
    std::vector<char> seen(kv->n_ctx, 0);
    for (int t = 0; t < nt; ++t) {
      if (seen[pos[t]]) return -1;
      seen[pos[t]] = 1;
    }
  }
  const orc_hparams& hp = m->hp;
  for (int t = 0; t < nt; ++t)
    if (ids[t] < 0 || ids[t] >= hp.n_vocab) return -3;
  if (orc_model_check(m) != 0) return -4;

  const int64_t H = hp.n_embd, nh = hp.n_head, nkv = hp.n_head_kv, hd = hp.head_dim;
  const int64_t q = nh * hd, kvw = nkv * hd, F = hp.n_ff;
  const int64_t nbH = (H + 31) / 32, nbq = (q + 31) / 32, nbF = (F + 31) / 32;

  std::vector<float> c((int64_t)kv->n_ctx * (hd / 2)), s((int64_t)kv->n_ctx * (hd / 2));
  rope_table(kv->n_ctx, (int)hd, hp.rope_theta, c.data(), s.data());

  /* embedding: one dequantized tok_embd row per id ([P05] section 2.5, embed GetRows) */
  std::vector<float> h((int64_t)nt * H);
  for (int t = 0; t < nt; ++t)
    for (int64_t k = 0; k < H; ++k)
      h[t * H + k] = f16_to_f32(m->tok_embd.d[(int64_t)ids[t] * nbH + k / 32]) *
                     (float)m->tok_embd.q[(int64_t)ids[t] * nbH * 32 + k];
  if (hidden) std::memcpy(hidden, h.data(), sizeof(float) * nt * H);

  std::vector<float> xn, Q, Kt, Vt, att, o, g, u, sw, dn;
  std::vector<int8_t> xq;
  std::vector<uint16_t> xd;
  int rows = nt; /* rows of h still carried */
  for (int l = 0; l < hp.n_layer; ++l) {
    OrcLayer& L = m->layers[l];
    /* attn_norm -> Q8_0 */
    xn.assign((int64_t)rows * H, 0.0f);
    for (int t = 0; t < rows; ++t) rmsnorm_row(&h[t * H], L.attn_norm.data(), H, hp.rms_eps, &xn[t * H]);
    xq.assign((int64_t)rows * nbH * 32, 0); xd.assign((int64_t)rows * nbH, 0);
    orc_q8_quantize(xn.data(), rows, H, xq.data(), xd.data());
    /* Q, K, V with bias */
    Q.assign((int64_t)rows * q, 0); Kt.assign((int64_t)rows * kvw, 0); Vt.assign((int64_t)rows * kvw, 0);
    matmul_q8(xq.data(), xd.data(), rows, L.wq, L.bq.empty() ? nullptr : L.bq.data(), Q.data());
    matmul_q8(xq.data(), xd.data(), rows, L.wk, L.bk.empty() ? nullptr : L.bk.data(), Kt.data());
    matmul_q8(xq.data(), xd.data(), rows, L.wv, L.bv.empty() ? nullptr : L.bv.data(), Vt.data());
    if (hp.qk_norm) {
      /* reading R8: per-head RMSNorm of Q and K, after the bias, before RoPE */
      std::vector<float> tmp(hd);
      for (int t = 0; t < rows; ++t) {
        for (int64_t hh = 0; hh < nh; ++hh) {
          float* x = &Q[t * q + hh * hd];
          rmsnorm_row(x, L.q_norm.data(), hd, hp.rms_eps, tmp.data());
          std::memcpy(x, tmp.data(), sizeof(float) * hd);
        }
        for (int64_t hh = 0; hh < nkv; ++hh) {
          float* x = &Kt[t * kvw + hh * hd];
          rmsnorm_row(x, L.k_norm.data(), hd, hp.rms_eps, tmp.data());
          std::memcpy(x, tmp.data(), sizeof(float) * hd);
        }
      }
    }
    rope_apply(Q.data(), rows, (int)nh, (int)hd, pos, c.data(), s.data());
    rope_apply(Kt.data(), rows, (int)nkv, (int)hd, pos, c.data(), s.data());
    /* kvcache_store: position p writes row p ([P09] section 2.2) */
    for (int t = 0; t < rows; ++t) {
      std::memcpy(&kv->k[l][(int64_t)pos[t] * kvw], &Kt[t * kvw], sizeof(float) * kvw);
      std::memcpy(&kv->v[l][(int64_t)pos[t] * kvw], &Vt[t * kvw], sizeof(float) * kvw);
    }
    /* attention over the region, all rows */
    att.assign((int64_t)rows * q, 0.0f);
    attention(Q.data(), rows, pos, kv->k[l].data(), kv->v[l].data(), (int)nh, (int)nkv, (int)hd, att.data());
    xq.assign((int64_t)rows * nbq * 32, 0); xd.assign((int64_t)rows * nbq, 0);
    orc_q8_quantize(att.data(), rows, q, xq.data(), xd.data());
    o.assign((int64_t)rows * H, 0.0f);
    matmul_q8(xq.data(), xd.data(), rows, L.wo, nullptr, o.data());
    /* tail rows on the last layer ([P05] section 2.8) */
    if (l == hp.n_layer - 1 && n_out < rows) {
      const int first = rows - n_out;
      std::vector<float> ht((int64_t)n_out * H), ot((int64_t)n_out * H);
      std::memcpy(ht.data(), &h[(int64_t)first * H], sizeof(float) * n_out * H);
      std::memcpy(ot.data(), &o[(int64_t)first * H], sizeof(float) * n_out * H);
      h.swap(ht); o.swap(ot);
      rows = n_out;
    }
    for (int64_t i = 0; i < (int64_t)rows * H; ++i) h[i] = h[i] + o[i];
    /* FFN */
    xn.assign((int64_t)rows * H, 0.0f);
    for (int t = 0; t < rows; ++t) rmsnorm_row(&h[t * H], L.ffn_norm.data(), H, hp.rms_eps, &xn[t * H]);
    xq.assign((int64_t)rows * nbH * 32, 0); xd.assign((int64_t)rows * nbH, 0);
    orc_q8_quantize(xn.data(), rows, H, xq.data(), xd.data());
    g.assign((int64_t)rows * F, 0); u.assign((int64_t)rows * F, 0);
    matmul_q8(xq.data(), xd.data(), rows, L.wg, nullptr, g.data());
    matmul_q8(xq.data(), xd.data(), rows, L.wu, nullptr, u.data());
    sw.assign((int64_t)rows * F, 0);
    for (int64_t i = 0; i < (int64_t)rows * F; ++i) sw[i] = swiglu(g[i], u[i]);
    xq.assign((int64_t)rows * nbF * 32, 0); xd.assign((int64_t)rows * nbF, 0);
    orc_q8_quantize(sw.data(), rows, F, xq.data(), xd.data());
    dn.assign((int64_t)rows * H, 0);
    matmul_q8(xq.data(), xd.data(), rows, L.wd, nullptr, dn.data());
    for (int64_t i = 0; i < (int64_t)rows * H; ++i) h[i] = h[i] + dn[i];
    if (hidden) std::memcpy(hidden + (int64_t)(l + 1) * nt * H, h.data(), sizeof(float) * rows * H);
  }
  /* final norm + lm_head on the carried rows */
  xn.assign((int64_t)rows * H, 0.0f);
  for (int t = 0; t < rows; ++t) rmsnorm_row(&h[t * H], m->out_norm.data(), H, hp.rms_eps, &xn[t * H]);
  xq.assign((int64_t)rows * nbH * 32, 0); xd.assign((int64_t)rows * nbH, 0);
  orc_q8_quantize(xn.data(), rows, H, xq.data(), xd.data());
  const QMat& wout = hp.tied_embeddings ? m->tok_embd : m->output;
  std::vector<float> lg((int64_t)rows * hp.n_vocab);
  matmul_q8(xq.data(), xd.data(), rows, wout, nullptr, lg.data());
  std::memcpy(logits, lg.data() + (int64_t)(rows - n_out) * hp.n_vocab,
              sizeof(float) * n_out * hp.n_vocab);
  return 0;
}

/* Index of the largest value; ties go to the lowest index (reading R7). */
int64_t orc_argmax(const float* x, int64_t n) {
  int64_t best = 0;
  for (int64_t i = 1; i < n; ++i)
    if (x[i] > x[best]) best = i;
  return best;
}

}  // extern "C"
