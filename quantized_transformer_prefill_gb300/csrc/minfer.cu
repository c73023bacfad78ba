// minfer.cu -- host side of the prefill library: weight loading and repacking,
// KV regions, the launch sequence of one prefill forward (recorded once per
// shape as a CUDA graph and replayed), and the C ABI of include/minfer.h.
//
// The forward follows the node list of "05 · Graph build — the IR and the
// builder", section 2.5, with the tail rows of section 2.8 and the call
// contract of "09 · Prefill: the first forward", section 3.2 (preflight,
// fill inputs, execute, one copy of the logits out):
//
//   validate ids/positions                          (device status word)
//   h = embed(ids)
//   x = Q8_0(rmsnorm(h) * attn_norm[0])
//   per layer l < L-1:
//     [Q|K|V] = x . Wqkv + b        tensor-core GEMM (split-K partials)
//     RoPE(Q, K); K/V rows pos[t]  <- K, V
//     a = attention(Q, regions)     all rows
//     o = Q8_0(a) . Wo              GEMM
//     h += o; x = Q8_0(rmsnorm(h) * ffn_norm)
//     s = Q8_0(silu(x.Wg) * x.Wu)   GEMM with SwiGLU + quantize epilogue
//     d = s . Wd                    GEMM
//     h += d; x = Q8_0(rmsnorm(h) * attn_norm[l+1])
//   last layer: QKV GEMM, RoPE and KV store on all rows (the regions must hold
//   every prompt row); attention, o-projection, FFN, final norm and lm_head
//   on the last row only, as one-row int8 GEMVs.  Rows other than the last
//   never reach the logits ("05 · Graph build", section 2.8), so cutting
//   them before the last attention changes no output.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/minfer.h"
#include "kernels.h"

using namespace minfer;

namespace {

#define CK(x)                                                   \
  do {                                                          \
    cudaError_t e_ = (x);                                       \
    if (e_ != cudaSuccess) {                                    \
      record_cuda_error(e_, #x, __LINE__);                      \
      return e_ == cudaErrorMemoryAllocation ? MINFER_ERR_OOM : MINFER_ERR_CUDA; \
    }                                                           \
  } while (0)

thread_local char g_last_error[512] = "";

void record_cuda_error(cudaError_t e, const char* what, int line) {
  snprintf(g_last_error, sizeof g_last_error, "%s (%s) at minfer.cu:%d: %s",
           cudaGetErrorName(e), cudaGetErrorString(e), line, what);
}

int64_t rup(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

template <typename T>
int dalloc(T** p, size_t count) {
  *p = nullptr;
  if (count == 0) return MINFER_OK;
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(p), count * sizeof(T));
  if (e != cudaSuccess) {
    record_cuda_error(e, "cudaMalloc", __LINE__);
    *p = nullptr;
    return MINFER_ERR_OOM;
  }
  e = cudaMemset(*p, 0, count * sizeof(T));
  if (e != cudaSuccess) {
    record_cuda_error(e, "cudaMemset", __LINE__);
    return MINFER_ERR_CUDA;
  }
  return MINFER_OK;
}

template <typename T>
void dfree(T*& p) {
  if (p) cudaFree(p);
  p = nullptr;
}

// A weight in the tensor-core layout.
struct GemmW {
  __half* codes = nullptr;
  float* scales = nullptr;
  int64_t rows = 0, rows_pad = 0;
  int nb = 0;
  GemmOperand op() const {
    GemmOperand o;
    o.codes = codes;
    o.scales = scales;
    o.rows = rows;
    o.rows_pad = rows_pad;
    o.nb = nb;
    return o;
  }
  int alloc(int64_t r, int n_blocks) {
    rows = r;
    rows_pad = rup(r, 128);
    nb = n_blocks;
    int rc = dalloc(&codes, (size_t)rows * nb * 32);
    if (rc) return rc;
    return dalloc(&scales, (size_t)nb * rows_pad);
  }
  void release() {
    dfree(codes);
    dfree(scales);
  }
};

// A weight in the one-row GEMV layout.
struct GemvW {
  int8_t* q = nullptr;
  float* s = nullptr;
  int64_t rows = 0;
  int nb = 0;
  int alloc(int64_t r, int n_blocks) {
    rows = r;
    nb = n_blocks;
    int rc = dalloc(&q, (size_t)rows * nb * 32);
    if (rc) return rc;
    return dalloc(&s, (size_t)rows * nb);
  }
  void release() {
    dfree(q);
    dfree(s);
  }
};

struct Layer {
  float* attn_norm = nullptr;
  float* ffn_norm = nullptr;
  float* bqkv = nullptr;                              // zero when the model has no biases
  float* q_norm = nullptr, *k_norm = nullptr;  // Qwen3 QK-norm weights [hd]
  GemmW wqkv, wo, wgu, wd;  // the last layer's o/FFN serve calls that want several logits rows
  // one-row (GEMV) layout of every matrix: the last layer's tail and
  // single-token calls (decode-shaped prefill)
  GemvW wqkv_v, wo_v, wgu_v, wd_v;
};

// Activation buffers for up to max_nt rows.
struct Workspace {
  int max_nt = 0;
  int32_t* ids = nullptr;
  int32_t* pos = nullptr;
  float* h = nullptr;        // [nt][H]
  __half* xa = nullptr;      // [nt][kx] codes (norm outputs and attention output)
  float* xa_s = nullptr;     // [nbx][ntp]
  __half* xf = nullptr;      // [nt][Fp] SwiGLU codes
  float* xf_s = nullptr;     // [nbF][ntp]
  float* part = nullptr;     // [splits][nt][max(qkvN, H)]
  int64_t part_stride = 0;
  float* qrot = nullptr;     // [nt][q]
  __half* qpl = nullptr;     // [2][nt][q] fp16 hi/lo of qrot (tensor-core attention)
  float* att = nullptr;      // [nt][q]
  float* h_last = nullptr;   // [H]
  int8_t* t_q = nullptr;     // [max kpad] one-row codes
  float* t_s = nullptr;      // [max nb]
  int8_t* t_q2 = nullptr;    // [Fp] one-row SwiGLU codes
  float* t_s2 = nullptr;     // [nbF]
  unsigned* tickets = nullptr;  // [kTickets] zero-initialized counters of the fused one-row norms
  float* logits = nullptr;   // [logits_rows][V]
  int logits_rows = 0;
  float* lm_out = nullptr;   // [logits_rows][V]: lm_head GEMM output before the status-gated copy
  int ntp = 0;
  void release() {
    dfree(ids); dfree(pos); dfree(h); dfree(xa); dfree(xa_s); dfree(xf); dfree(xf_s);
    dfree(part); dfree(qrot); dfree(qpl); dfree(att); dfree(h_last); dfree(t_q); dfree(t_s);
    dfree(t_q2); dfree(t_s2); dfree(tickets);
    dfree(logits); dfree(lm_out);
    logits_rows = 0;
    max_nt = 0;
  }
};

constexpr int kMaxSplits = 8;
// tickets of the fused norms of the one-row o and down GEMVs
constexpr int kTicketNormO = 0, kTicketNormDown = 1;
constexpr int kTickets = 2;

enum KClass : int {
  kKValidate, kKEmbed, kKRowQuant, kKGemmQKV, kKRope, kKAttn, kKGemmO, kKGemmGU, kKGemmDown,
  kKTailGemv, kKLmHead, kNumKClass
};
const char* kClassNames[kNumKClass] = {
    "validate", "embed", "rmsnorm_quant", "gemm_qkv", "rope_kv_store", "attention", "gemm_o",
    "gemm_gate_up_swiglu", "gemm_down", "tail_gemv", "lm_head_gemv"};

}  // namespace

struct minfer_kv {
  minfer_model* m = nullptr;
  int n_ctx = 0;
  float* regions = nullptr;  // [L][2][n_ctx][kvw]
  __half* shadow = nullptr;  // [L][4][n_ctx][kvw]: fp16 hi/lo of K and V, read by attention
  __half* vt = nullptr;      // [L][2][kvw][vt_ld]: fp16 hi/lo of V transposed (key-major)
  int64_t vt_ld = 0;         // n_ctx rounded up to 64
  float* cos_t = nullptr;    // [n_ctx][hd/2]
  float* sin_t = nullptr;
  uint32_t* seen = nullptr;  // n_ctx bits (duplicate-position check)
  float* k(int l) const;
  float* v(int l) const;
  __half* plane(int l, int i) const;
  __half* vtp(int l, int i) const { return vt + ((int64_t)l * 2 + i) * m_kvw * vt_ld; }
  int64_t m_kvw = 0;
};

struct minfer_model {
  int device = 0;
  int num_sms = 148;
  minfer_hparams hp{};
  int64_t H = 0, q = 0, kvw = 0, F = 0, Fp = 0, V = 0, qkvN = 0;
  int nbH = 0, nbq = 0, nbF = 0;
  cudaStream_t stream = nullptr;
  GemvW tok_embd, output;
  GemmW lm_gemm;  // the lm_head in the tensor-core layout, built on the first n_out > 1 call
  float* out_norm = nullptr;
  std::vector<Layer> layers;
  std::map<std::string, bool> have;
  bool finalized = false;
  Workspace ws;
  int* d_status = nullptr;
  int* h_status = nullptr;  // pinned
  // staging for loads
  void* stage = nullptr;
  size_t stage_bytes = 0;
  int8_t* stage_q = nullptr;
  uint16_t* stage_d = nullptr;
  size_t stage_q_bytes = 0;
  // graph cache
  struct GraphKey {
    int nt = 0, n_out = 1;
    const minfer_kv* kv = nullptr;
    const void *ids = nullptr, *pos = nullptr, *logits = nullptr;
    bool profile = false;
    bool operator==(const GraphKey& o) const {
      return nt == o.nt && n_out == o.n_out && kv == o.kv && ids == o.ids && pos == o.pos &&
             logits == o.logits && profile == o.profile;
    }
  };
  GraphKey gkey;
  cudaGraphExec_t gexec = nullptr;
  cudaGraph_t graph = nullptr;
  // profiling
  bool profile = false;
  std::vector<cudaEvent_t> ev;  // pairs per launch
  std::vector<int> ev_class;
  int ev_used = 0;
  double prof_ms[kNumKClass] = {};
  int64_t prof_n[kNumKClass] = {};
  // dumps
  float* dump_host = nullptr;
  int dump_max_nt = 0;
  int last_device_status = 0;
  // test hook of the bounded-wait failure path (minfer_debug_fault)
  int fault_layer = -1;
  uint64_t fault_wait_ns = 0;
  bool debug_f32 = false;  // also write the f32 attention output (debug reads)
  // stage capture of one layer (debug): copies of that layer's intermediates
  int dbg_layer = -1;
  int dbg_nt = 0;
  bool dump_on = false;  // this call copies hidden states to dump_host
  std::map<std::string, std::pair<void*, size_t>> dbg;  // name -> (device buffer, bytes)
};

float* minfer_kv::k(int l) const {
  return regions + ((int64_t)l * 2 + 0) * n_ctx * m->kvw;
}
float* minfer_kv::v(int l) const {
  return regions + ((int64_t)l * 2 + 1) * n_ctx * m->kvw;
}
__half* minfer_kv::plane(int l, int i) const {
  return shadow + ((int64_t)l * 4 + i) * n_ctx * m->kvw;
}

namespace {

std::mutex g_mu;

// ------------------------------------------------------------------ loading

int ensure_stage(minfer_model* m, size_t bytes, size_t q_elems, size_t nblocks) {
  if (bytes > m->stage_bytes) {
    if (m->stage) cudaFree(m->stage);
    m->stage = nullptr;
    CK(cudaMalloc(&m->stage, bytes));
    m->stage_bytes = bytes;
  }
  if (q_elems > m->stage_q_bytes) {
    dfree(m->stage_q);
    dfree(m->stage_d);
    int rc = dalloc(&m->stage_q, q_elems);
    if (rc) return rc;
    rc = dalloc(&m->stage_d, std::max<size_t>(nblocks, q_elems / 32));
    if (rc) return rc;
    m->stage_q_bytes = q_elems;
  }
  return MINFER_OK;
}

// Upload a matrix [ne1][ne0] (F32 or Q8_0 blocks) and leave its int8 codes
// [ne1][nb*32] and fp16 bits [ne1][nb] in the model's staging buffers.
int stage_matrix(minfer_model* m, const minfer_tensor* t) {
  const int64_t nb = (t->ne0 + 31) / 32;
  const size_t q_elems = (size_t)t->ne1 * nb * 32;
  const size_t in_bytes =
      t->type == MINFER_F32 ? (size_t)t->ne0 * t->ne1 * 4 : (size_t)t->ne1 * nb * 34;
  int rc = ensure_stage(m, in_bytes, q_elems, (size_t)t->ne1 * nb);
  if (rc) return rc;
  CK(cudaMemcpyAsync(m->stage, t->data, in_bytes, cudaMemcpyHostToDevice, m->stream));
  if (t->type == MINFER_F32)
    CK(quantize_rows_launch(static_cast<const float*>(m->stage), t->ne1, t->ne0, m->stage_q,
                            m->stage_d, m->stream));
  else
    CK(unpack_q8_0_launch(static_cast<const uint8_t*>(m->stage), t->ne1, t->ne0, m->stage_q,
                          m->stage_d, m->stream));
  return MINFER_OK;
}

int to_gemm(minfer_model* m, int64_t rows, int nb, GemmW& w, int64_t row0, int interleave,
            int which) {
  RepackArgs r;
  r.q = m->stage_q;
  r.dbits = m->stage_d;
  r.rows = rows;
  r.nb = nb;
  r.dst_codes = w.codes;
  r.dst_scales = w.scales;
  r.dst_rows_pad = w.rows_pad;
  r.dst_row0 = row0;
  r.interleave = interleave;
  r.which = which;
  CK(repack_gemm_launch(r, m->stream));
  return MINFER_OK;
}

int to_gemv(minfer_model* m, int64_t rows, int nb, GemvW& w, int64_t row0, int interleave = 0,
            int which = 0) {
  CK(repack_gemv_launch(m->stage_q, m->stage_d, rows, nb, w.q + row0 * nb * 32, w.s + row0 * nb,
                        interleave, which, m->stream));
  return MINFER_OK;
}

int upload_vec(minfer_model* m, float* dst, const minfer_tensor* t) {
  CK(cudaMemcpyAsync(dst, t->data, (size_t)t->ne0 * 4, cudaMemcpyHostToDevice, m->stream));
  return MINFER_OK;
}

bool parse_layer(const char* name, int* layer, std::string* kind) {
  if (strncmp(name, "blk.", 4) != 0) return false;
  char* end = nullptr;
  long l = strtol(name + 4, &end, 10);
  if (!end || *end != '.' || end == name + 4) return false;
  *layer = (int)l;
  *kind = std::string(end + 1);
  return true;
}

int model_alloc(minfer_model* m) {
  const auto& hp = m->hp;
  m->H = hp.n_embd;
  m->q = (int64_t)hp.n_head * hp.head_dim;
  m->kvw = (int64_t)hp.n_head_kv * hp.head_dim;
  m->F = hp.n_ff;
  m->V = hp.n_vocab;
  m->nbH = (int)((m->H + 31) / 32);
  m->nbq = (int)((m->q + 31) / 32);
  m->nbF = (int)((m->F + 31) / 32);
  m->Fp = (int64_t)m->nbF * 32;
  m->qkvN = m->q + 2 * m->kvw;
  int rc;
  if ((rc = m->tok_embd.alloc(m->V, m->nbH))) return rc;
  if (!hp.tied_embeddings && (rc = m->output.alloc(m->V, m->nbH))) return rc;
  if ((rc = dalloc(&m->out_norm, m->H))) return rc;
  m->layers.resize(hp.n_layer);
  for (int l = 0; l < hp.n_layer; ++l) {
    Layer& L = m->layers[l];
    const bool last = l == hp.n_layer - 1;
    if ((rc = dalloc(&L.attn_norm, m->H)) || (rc = dalloc(&L.ffn_norm, m->H)) ||
        (rc = dalloc(&L.bqkv, m->qkvN)))
      return rc;
    if (hp.qk_norm &&
        ((rc = dalloc(&L.q_norm, hp.head_dim)) || (rc = dalloc(&L.k_norm, hp.head_dim))))
      return rc;
    if ((rc = L.wqkv.alloc(m->qkvN, m->nbH)) || (rc = L.wo.alloc(m->H, m->nbq)) ||
        (rc = L.wgu.alloc(2 * m->Fp, m->nbH)) || (rc = L.wd.alloc(m->H, m->nbF)))
      return rc;
    if ((rc = L.wqkv_v.alloc(m->qkvN, m->nbH)) || (rc = L.wo_v.alloc(m->H, m->nbq)) ||
        (rc = L.wgu_v.alloc(2 * m->Fp, m->nbH)) || (rc = L.wd_v.alloc(m->H, m->nbF)))
      return rc;
  }
  if ((rc = dalloc(&m->d_status, 4))) return rc;
  CK(cudaMallocHost(&m->h_status, 4 * sizeof(int)));
  return MINFER_OK;
}

void model_release(minfer_model* m) {
  m->lm_gemm.release();
  for (auto& kv : m->dbg)
    if (kv.second.first) cudaFree(kv.second.first);
  m->dbg.clear();
  if (m->gexec) cudaGraphExecDestroy(m->gexec);
  if (m->graph) cudaGraphDestroy(m->graph);
  for (auto e : m->ev) cudaEventDestroy(e);
  m->tok_embd.release();
  m->output.release();
  dfree(m->out_norm);
  for (auto& L : m->layers) {
    dfree(L.attn_norm); dfree(L.ffn_norm); dfree(L.bqkv); dfree(L.q_norm); dfree(L.k_norm);
    L.wqkv.release(); L.wo.release(); L.wgu.release(); L.wd.release();
    L.wqkv_v.release(); L.wo_v.release(); L.wgu_v.release(); L.wd_v.release();
  }
  m->ws.release();
  dfree(m->d_status);
  if (m->h_status) cudaFreeHost(m->h_status);
  if (m->stage) cudaFree(m->stage);
  dfree(m->stage_q);
  dfree(m->stage_d);
  if (m->stream) cudaStreamDestroy(m->stream);
}

int set_tensor(minfer_model* m, const minfer_tensor* t) {
  if (!t || !t->name || !t->data) return MINFER_ERR_ARG;
  const auto& hp = m->hp;
  const std::string name(t->name);
  const bool is_f32 = t->type == MINFER_F32, is_q8 = t->type == MINFER_Q8_0;
  if (!is_f32 && !is_q8) return MINFER_ERR_SHAPE;
  auto vec_ok = [&](int64_t n) { return is_f32 && t->ne0 == n && t->ne1 == 1; };
  auto mat_ok = [&](int64_t in, int64_t out) { return t->ne0 == in && t->ne1 == out; };
  int rc = MINFER_OK;
  if (name == "token_embd.weight") {
    if (!mat_ok(m->H, m->V)) return MINFER_ERR_SHAPE;
    if ((rc = stage_matrix(m, t)) || (rc = to_gemv(m, m->V, m->nbH, m->tok_embd, 0))) return rc;
  } else if (name == "output.weight") {
    if (hp.tied_embeddings || !mat_ok(m->H, m->V)) return MINFER_ERR_SHAPE;
    if ((rc = stage_matrix(m, t)) || (rc = to_gemv(m, m->V, m->nbH, m->output, 0))) return rc;
  } else if (name == "output_norm.weight") {
    if (!vec_ok(m->H)) return MINFER_ERR_SHAPE;
    if ((rc = upload_vec(m, m->out_norm, t))) return rc;
  } else {
    int l;
    std::string k;
    if (!parse_layer(t->name, &l, &k) || l < 0 || l >= hp.n_layer) return MINFER_ERR_SHAPE;
    Layer& L = m->layers[l];
    const bool last = l == hp.n_layer - 1;
    if (k == "attn_norm.weight") {
      if (!vec_ok(m->H)) return MINFER_ERR_SHAPE;
      rc = upload_vec(m, L.attn_norm, t);
    } else if (k == "ffn_norm.weight") {
      if (!vec_ok(m->H)) return MINFER_ERR_SHAPE;
      rc = upload_vec(m, L.ffn_norm, t);
    } else if (hp.qk_norm && (k == "attn_q_norm.weight" || k == "attn_k_norm.weight")) {
      if (!vec_ok(hp.head_dim)) return MINFER_ERR_SHAPE;
      rc = upload_vec(m, k == "attn_q_norm.weight" ? L.q_norm : L.k_norm, t);
    } else if (k == "attn_q.bias" || k == "attn_k.bias" || k == "attn_v.bias") {
      const int64_t n = k == "attn_q.bias" ? m->q : m->kvw;
      const int64_t off = k == "attn_q.bias" ? 0 : (k == "attn_k.bias" ? m->q : m->q + m->kvw);
      if (!vec_ok(n)) return MINFER_ERR_SHAPE;
      CK(cudaMemcpyAsync(L.bqkv + off, t->data, (size_t)n * 4, cudaMemcpyHostToDevice, m->stream));
    } else if (k == "attn_q.weight" || k == "attn_k.weight" || k == "attn_v.weight") {
      const int64_t n = k == "attn_q.weight" ? m->q : m->kvw;
      const int64_t off = k == "attn_q.weight" ? 0 : (k == "attn_k.weight" ? m->q : m->q + m->kvw);
      if (!mat_ok(m->H, n)) return MINFER_ERR_SHAPE;
      if ((rc = stage_matrix(m, t)) || (rc = to_gemm(m, n, m->nbH, L.wqkv, off, 0, 0)) ||
          (rc = to_gemv(m, n, m->nbH, L.wqkv_v, off)))
        return rc;
    } else if (k == "attn_output.weight") {
      if (!mat_ok(m->q, m->H)) return MINFER_ERR_SHAPE;
      if ((rc = stage_matrix(m, t))) return rc;
      if ((rc = to_gemm(m, m->H, m->nbq, L.wo, 0, 0, 0))) return rc;
      rc = to_gemv(m, m->H, m->nbq, L.wo_v, 0);
    } else if (k == "ffn_gate.weight" || k == "ffn_up.weight") {
      const int which = k == "ffn_gate.weight" ? 0 : 1;
      if (!mat_ok(m->H, m->F)) return MINFER_ERR_SHAPE;
      if ((rc = stage_matrix(m, t))) return rc;
      if ((rc = to_gemm(m, m->F, m->nbH, L.wgu, 0, 1, which))) return rc;
      rc = to_gemv(m, m->F, m->nbH, L.wgu_v, 0, 1, which);
    } else if (k == "ffn_down.weight") {
      if (!mat_ok(m->F, m->H)) return MINFER_ERR_SHAPE;
      if ((rc = stage_matrix(m, t))) return rc;
      if ((rc = to_gemm(m, m->H, m->nbF, L.wd, 0, 0, 0))) return rc;
      rc = to_gemv(m, m->H, m->nbF, L.wd_v, 0);
    } else {
      return MINFER_ERR_SHAPE;
    }
    if (rc) return rc;
  }
  CK(cudaStreamSynchronize(m->stream));  // host data may be freed on return
  m->have[name] = true;
  return MINFER_OK;
}

std::vector<std::string> required_names(const minfer_hparams& hp) {
  std::vector<std::string> v = {"token_embd.weight", "output_norm.weight"};
  if (!hp.tied_embeddings) v.push_back("output.weight");
  const char* kinds[] = {"attn_norm.weight", "attn_q.weight", "attn_k.weight", "attn_v.weight",
                         "attn_output.weight", "ffn_norm.weight", "ffn_gate.weight",
                         "ffn_up.weight", "ffn_down.weight"};
  // Qwen2: Q/K/V biases; Qwen3: the QK-norm weights (biases optional)
  const char* qwen2[] = {"attn_q.bias", "attn_k.bias", "attn_v.bias"};
  const char* qwen3[] = {"attn_q_norm.weight", "attn_k_norm.weight"};
  for (int l = 0; l < hp.n_layer; ++l) {
    const std::string b = "blk." + std::to_string(l) + ".";
    for (const char* k : kinds) v.push_back(b + k);
    if (hp.qk_norm)
      for (const char* k : qwen3) v.push_back(b + k);
    else
      for (const char* k : qwen2) v.push_back(b + k);
  }
  return v;
}

// ------------------------------------------------------------------ workspace

int ensure_workspace(minfer_model* m, int nt) {
  Workspace& w = m->ws;
  if (nt <= w.max_nt) return MINFER_OK;
  if (m->gexec) {
    cudaGraphExecDestroy(m->gexec);
    m->gexec = nullptr;
  }
  if (m->graph) {
    cudaGraphDestroy(m->graph);
    m->graph = nullptr;
  }
  w.release();
  const int64_t ntp = rup(nt, 128);
  const int64_t kx = std::max<int64_t>((int64_t)m->nbH, m->nbq) * 32;
  const int nbx = std::max(m->nbH, m->nbq);
  const int64_t pw = std::max(m->qkvN, m->H);
  int rc;
  if ((rc = dalloc(&w.ids, nt)) || (rc = dalloc(&w.pos, nt)) || (rc = dalloc(&w.h, nt * m->H)) ||
      (rc = dalloc(&w.xa, ntp * kx)) || (rc = dalloc(&w.xa_s, (size_t)nbx * ntp)) ||
      (rc = dalloc(&w.xf, ntp * m->Fp)) || (rc = dalloc(&w.xf_s, (size_t)m->nbF * ntp)) ||
      (rc = dalloc(&w.part, (size_t)kMaxSplits * nt * pw)) || (rc = dalloc(&w.qrot, nt * m->q)) ||
      (rc = dalloc(&w.qpl, 2 * nt * m->q)) ||
      (rc = dalloc(&w.att, nt * m->q)) || (rc = dalloc(&w.h_last, m->H)) ||
      (rc = dalloc(&w.t_q, std::max<int64_t>(kx, m->Fp))) ||
      (rc = dalloc(&w.t_s, std::max(nbx, m->nbF))) || (rc = dalloc(&w.t_q2, m->Fp)) ||
      (rc = dalloc(&w.t_s2, m->nbF)) ||
      (rc = dalloc(&w.tickets, (size_t)kTickets)) ||
      (rc = dalloc(&w.logits, m->V)))
    return rc;
  w.logits_rows = 1;
  w.part_stride = (int64_t)nt * pw;
  w.ntp = (int)ntp;
  w.max_nt = nt;
  return MINFER_OK;
}

// ------------------------------------------------------------------ launch sequence

struct Launcher {
  minfer_model* m;
  cudaStream_t st;
  bool prof;
  int begin(int cls) {
    if (!prof) return MINFER_OK;
    if (m->ev_used + 2 > (int)m->ev.size()) {
      for (int i = 0; i < 64; ++i) {
        cudaEvent_t e;
        CK(cudaEventCreate(&e));
        m->ev.push_back(e);
        m->ev_class.push_back(-1);
      }
    }
    m->ev_class[m->ev_used] = cls;
    // external: under stream capture the record becomes a graph node that
    // records the event on every replay
    CK(cudaEventRecordWithFlags(m->ev[m->ev_used], st, cudaEventRecordExternal));
    return MINFER_OK;
  }
  int end() {
    if (!prof) return MINFER_OK;
    CK(cudaEventRecordWithFlags(m->ev[m->ev_used + 1], st, cudaEventRecordExternal));
    m->ev_used += 2;
    return MINFER_OK;
  }
};

#define LAUNCH(cls, call)            \
  do {                               \
    int rc_ = L.begin(cls);          \
    if (rc_) return rc_;             \
    CK(call);                        \
    if ((rc_ = L.end())) return rc_; \
  } while (0)

int gemm_call(minfer_model* m, Launcher& L, int cls, const GemmOperand& A, const GemmW& W,
              int64_t M, int epi, bool allow_split, float* out, int64_t ldo, __half* q_out,
              int64_t ldq, float* qs_out, int64_t ldqs, int* nsplit_out, bool fault = false) {
  GemmLaunch g;
  g.A = A;
  g.B = W.op();
  g.M = M;
  g.N = W.rows;
  g.epi = epi;
  g.plan = gemm_plan(M, W.rows, W.nb, m->num_sms, allow_split);
  g.plan.splits = std::min(g.plan.splits, kMaxSplits);
  g.out = out;
  g.ldo = ldo;
  g.split_stride = m->ws.part_stride;
  g.q_out = q_out;
  g.ldq = ldq;
  g.qs_out = qs_out;
  g.ldqs = ldqs;
  g.n_out_cols = m->Fp;
  g.err = m->d_status + 1;
  g.b_static = true;  // the model's weights, uploaded (and synchronized) at load
  if (m->fault_layer >= 0) {
    g.wait_ns = m->fault_wait_ns;
    if (fault) g.skip_stage = 0;
  }
  GemmMaps maps;
  if (gemm_make_maps(g.A, g.B, g.plan.bn, &maps)) {
    snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled failed");
    return MINFER_ERR_CUDA;
  }
  // the kernel may round the split count; recompute it the same way
  const int stages = (W.nb + 1) / 2;
  int splits = std::max(1, std::min(g.plan.splits, stages));
  const int sps = (stages + splits - 1) / splits;
  splits = (stages + sps - 1) / sps;
  if (nsplit_out) *nsplit_out = splits;
  LAUNCH(cls, gemm_launch(g, maps, m->num_sms, L.st));
  return MINFER_OK;
}

// Copy `bytes` from src into the named stage-capture buffer (debug only).
int dbg_capture(minfer_model* m, cudaStream_t st, const char* name, const void* src, size_t bytes) {
  auto& e = m->dbg[name];
  if (e.second < bytes) {
    if (e.first) cudaFree(e.first);
    e.first = nullptr;
    e.second = 0;
    CK(cudaMalloc(&e.first, bytes));
    e.second = bytes;
  }
  CK(cudaMemcpyAsync(e.first, src, bytes, cudaMemcpyDeviceToDevice, st));
  return MINFER_OK;
}

// Capture a block-major scale plane [nb][ld] as [nb][ntp_call] (debug only).
int dbg_capture_scales(minfer_model* m, cudaStream_t st, const char* name, const float* src,
                       int nb, int64_t ld, int64_t ntp_call) {
  auto& e = m->dbg[name];
  const size_t bytes = (size_t)nb * ntp_call * 4;
  if (e.second < bytes) {
    if (e.first) cudaFree(e.first);
    e.first = nullptr;
    e.second = 0;
    CK(cudaMalloc(&e.first, bytes));
    e.second = bytes;
  }
  CK(cudaMemcpy2DAsync(e.first, ntp_call * 4, src, ld * 4, ntp_call * 4, nb,
                       cudaMemcpyDeviceToDevice, st));
  return MINFER_OK;
}

void dump_hidden(minfer_model* m, cudaStream_t st, int slot, const float* src, int rows) {
  if (!m->dump_on) return;
  float* dst = m->dump_host + (int64_t)slot * m->dump_max_nt * m->H;
  cudaMemcpyAsync(dst, src, (size_t)rows * m->H * 4, cudaMemcpyDeviceToHost, st);
}

// A single-token call (the decode shape, "09 · Prefill" section 2.3 with
// n_tokens = 1): every projection is a one-row GEMV over the int8 layout,
// which reads each weight byte once -- the work is bound by HBM, and the
// tensor-core GEMM would pad the one row to 128.
// ------------------------------------------------------------------ one-row stages
// Shared by single-token calls and the last row of a prompt: every projection
// is a GEMV over the one-row Q8_0 activation.

GemvArgs row_gemv(const minfer_model* m, const GemvW& W, int64_t N, int nb, const int8_t* xq,
                  const float* xs, float* y, const float* resid) {
  GemvArgs g;
  g.num_sms = m->num_sms;
  g.wq = W.q;
  g.ws = W.s;
  g.N = N;
  g.nb = nb;
  g.kpad = (int64_t)nb * 32;
  g.xq = xq;
  g.xs = xs;
  g.y = y;
  g.resid = resid;
  g.w_static = 1;  // the model's weights, uploaded (and synchronized) at load
  return g;
}

// y = resid + W.x, then RMSNorm(y) * norm_w quantized (Q8_0) into the one-row
// codes t_q/t_s: inside the GEMV's last CTA where the shape allows, else by
// the row kernel after it.
int row_gemv_norm(minfer_model* m, Launcher& L, GemvArgs g, const float* norm_w, int ticket,
                  cudaStream_t st) {
  Workspace& w = m->ws;
  if (gemv_norm_fusable(g.N, g.y, norm_w, w.t_q)) {
    g.norm_w = norm_w;
    g.eps = m->hp.rms_eps;
    g.q8 = w.t_q;
    g.s8 = w.t_s;
    g.ticket = w.tickets + ticket;
    LAUNCH(kKTailGemv, gemv_launch(g, st));
    return MINFER_OK;
  }
  LAUNCH(kKTailGemv, gemv_launch(g, st));
  RowQuantArgs r;
  r.h = g.y;
  r.norm_w = norm_w;
  r.eps = m->hp.rms_eps;
  r.rows = 1;
  r.n = g.N;
  r.q8 = w.t_q;
  r.s8 = w.t_s;
  LAUNCH(kKRowQuant, row_quant_launch(r, st));
  return MINFER_OK;
}

// gate/up GEMV with the SwiGLU and its Q8_0 in the same kernel: t_q/t_s in,
// t_q2/t_s2 out.
int row_gemv_swiglu(minfer_model* m, Launcher& L, const GemvW& W, cudaStream_t st) {
  Workspace& w = m->ws;
  GemvArgs g = row_gemv(m, W, 2 * m->Fp, m->nbH, w.t_q, w.t_s, nullptr, nullptr);
  g.swiglu = 1;
  g.q8 = w.t_q2;
  g.s8 = w.t_s2;
  LAUNCH(kKTailGemv, gemv_launch(g, st));
  return MINFER_OK;
}

// The one-row attention kernel's inputs on top of the tiled kernel's.
void row_attention_args(const minfer_kv* kv, int l, AttnArgs* at) {
  at->kreg = kv->k(l);
  at->vreg = kv->v(l);
}

int enqueue_decode(minfer_model* m, minfer_kv* kv, const int32_t* ids, const int32_t* pos,
                   float* logits, cudaStream_t st, bool prof, bool dumps) {
  const auto& hp = m->hp;
  Workspace& w = m->ws;
  Launcher L{m, st, prof};
  auto norm_quant = [&](const float* norm_w) -> int {
    RowQuantArgs r;
    r.h = w.h;
    r.norm_w = norm_w;
    r.eps = hp.rms_eps;
    r.rows = 1;
    r.n = m->H;
    r.q8 = w.t_q;
    r.s8 = w.t_s;
    LAUNCH(kKRowQuant, row_quant_launch(r, st));
    return MINFER_OK;
  };
  int rc;
  // stage capture of one layer (debug): one-row layouts, int8 codes + f32 scales
  auto cap_q8 = [&](const char* qname, const char* sname, int nb) -> int {
    int r;
    if ((r = dbg_capture(m, st, qname, w.t_q, (size_t)nb * 32)) ||
        (r = dbg_capture(m, st, sname, w.t_s, (size_t)nb * 4)))
      return r;
    return MINFER_OK;
  };
  CK(cudaMemsetAsync(m->d_status + 1, 0, sizeof(int), st));
  LAUNCH(kKValidate, validate_launch(ids, pos, 1, (int)m->V, kv->n_ctx, kv->seen, m->d_status, st));
  LAUNCH(kKEmbed, embed_launch(m->tok_embd.q, m->tok_embd.s, (int64_t)m->nbH * 32, m->nbH, ids, 1,
                               m->H, (int)m->V, w.h, st));
  if (dumps) dump_hidden(m, st, 0, w.h, 1);
  if ((rc = norm_quant(m->layers[0].attn_norm))) return rc;
  for (int l = 0; l < hp.n_layer; ++l) {
    Layer& Ly = m->layers[l];
    const bool cap = l == m->dbg_layer;
    if (cap) {
      for (auto& e : m->dbg)
        if (e.second.first) cudaFree(e.second.first);
      m->dbg.clear();
      m->dbg_nt = 1;
      if ((rc = dbg_capture(m, st, "h_in", w.h, (size_t)m->H * 4)) ||
          (rc = cap_q8("x_q8", "x_s8", m->nbH)))
        return rc;
    }
    {
      RopeStoreArgs r;
      r.partials = w.part;
      r.bias = Ly.bqkv;
      r.pos = pos;
      r.nt = 1;
      r.nh = hp.n_head;
      r.nkv = hp.n_head_kv;
      r.hd = hp.head_dim;
      r.n_ctx = kv->n_ctx;
      r.cos_t = kv->cos_t;
      r.sin_t = kv->sin_t;
      r.q_out = w.qrot;
      r.kreg = kv->k(l);
      r.vreg = kv->v(l);
      for (int i = 0; i < 4; ++i) r.shadow[i] = kv->plane(l, i);
      r.vt[0] = kv->vtp(l, 0);
      r.vt[1] = kv->vtp(l, 1);
      r.vt_ld = kv->vt_ld;
      r.status = m->d_status;
      if (hp.qk_norm) {
        r.q_norm = Ly.q_norm;
        r.k_norm = Ly.k_norm;
        r.eps = hp.rms_eps;
      }
      // Q|K|V sums -> w.part; RoPE/store in the same kernel unless QK-norm
      const GemvArgs gq = row_gemv(m, Ly.wqkv_v, m->qkvN, m->nbH, w.t_q, w.t_s, w.part, nullptr);
      if (!hp.qk_norm) {
        LAUNCH(kKTailGemv, gemv_rope_launch(gq, r, st));
      } else {
        LAUNCH(kKTailGemv, gemv_launch(gq, st));
        LAUNCH(kKRope, rope_store_launch(r, st));
      }
    }
    if (cap && (rc = dbg_capture(m, st, "qkv", w.part, (size_t)m->qkvN * 4))) return rc;
    {
      AttnArgs at;
      at.q = w.qrot;
      at.pos = pos;
      at.r0 = 0;
      at.r1 = 1;
      for (int i = 0; i < 4; ++i) at.shadow[i] = kv->plane(l, i);
      at.vt[0] = kv->vtp(l, 0);
      at.vt[1] = kv->vtp(l, 1);
      at.vt_ld = kv->vt_ld;
      at.nh = hp.n_head;
      at.nkv = hp.n_head_kv;
      at.hd = hp.head_dim;
      at.n_ctx = kv->n_ctx;
      at.nsplit = attention_nsplit(1, at.nkv, m->num_sms, at.nh / at.nkv);
      row_attention_args(kv, l, &at);
      at.kv_static_below = 1;  // rows below the token's position: earlier calls
      AttnOut ao;
      ao.f32 = (m->debug_f32 || cap) ? w.att : nullptr;
      ao.q8 = w.t_q;
      ao.s8 = w.t_s;
      LAUNCH(kKAttn, attention_launch(at, ao, st));
    }
    if (cap && ((rc = dbg_capture(m, st, "qrot", w.qrot, (size_t)m->q * 4)) ||
                (rc = dbg_capture(m, st, "att", w.att, (size_t)m->q * 4)) ||
                (rc = cap_q8("att_q8", "att_s8", m->nbq))))
      return rc;
    // o projection + residual, ffn_norm -> t_q/t_s
    if ((rc = row_gemv_norm(m, L, row_gemv(m, Ly.wo_v, m->H, m->nbq, w.t_q, w.t_s, w.h, w.h),
                            Ly.ffn_norm, kTicketNormO, st)))
      return rc;
    if (cap && (rc = dbg_capture(m, st, "h_mid", w.h, (size_t)m->H * 4))) return rc;
    if (cap && (rc = cap_q8("f_q8", "f_s8", m->nbH))) return rc;
    // gate/up + SwiGLU -> t_q2/t_s2
    if ((rc = row_gemv_swiglu(m, L, Ly.wgu_v, st))) return rc;
    if (cap && ((rc = dbg_capture(m, st, "s_q8", w.t_q2, (size_t)m->nbF * 32)) ||
                (rc = dbg_capture(m, st, "s_s8", w.t_s2, (size_t)m->nbF * 4))))
      return rc;
    // down + residual, the next norm (attn_norm of the next layer, or the output norm)
    if ((rc = row_gemv_norm(m, L, row_gemv(m, Ly.wd_v, m->H, m->nbF, w.t_q2, w.t_s2, w.h, w.h),
                            l + 1 < hp.n_layer ? m->layers[l + 1].attn_norm : m->out_norm,
                            kTicketNormDown, st)))
      return rc;
    if (cap && (rc = dbg_capture(m, st, "h_out", w.h, (size_t)m->H * 4))) return rc;
    if (dumps) dump_hidden(m, st, l + 1, w.h, 1);
  }
  const GemvW& out = hp.tied_embeddings ? m->tok_embd : m->output;
  GemvArgs g = row_gemv(m, out, m->V, m->nbH, w.t_q, w.t_s, logits, nullptr);
  g.status = m->d_status;
  LAUNCH(kKLmHead, gemv_launch(g, st));
  return MINFER_OK;
}

// Enqueue one forward.  ids/pos/logits are device pointers.
int enqueue_forward(minfer_model* m, minfer_kv* kv, const int32_t* ids, const int32_t* pos, int nt,
                    int n_out, float* logits, cudaStream_t st, bool prof, bool dumps) {
  if (nt == 1) return enqueue_decode(m, kv, ids, pos, logits, st, prof, dumps);
  const auto& hp = m->hp;
  Workspace& w = m->ws;
  Launcher L{m, st, prof};
  const int ntp = w.ntp;
  GemmOperand xa;
  xa.codes = w.xa;
  xa.scales = w.xa_s;
  xa.rows = nt;
  xa.rows_pad = ntp;
  xa.nb = m->nbH;
  GemmOperand xo = xa;  // attention output operand (K = q)
  xo.nb = m->nbq;
  GemmOperand xf;
  xf.codes = w.xf;
  xf.scales = w.xf_s;
  xf.rows = nt;
  xf.rows_pad = ntp;
  xf.nb = m->nbF;

  CK(cudaMemsetAsync(m->d_status + 1, 0, sizeof(int), st));
  LAUNCH(kKValidate, validate_launch(ids, pos, nt, (int)m->V, kv->n_ctx, kv->seen, m->d_status, st));
  LAUNCH(kKEmbed, embed_launch(m->tok_embd.q, m->tok_embd.s, (int64_t)m->nbH * 32, m->nbH, ids, nt,
                               m->H, (int)m->V, w.h, st));
  if (dumps) dump_hidden(m, st, 0, w.h, nt);
  {
    RowQuantArgs r;
    r.h = w.h;
    r.norm_w = m->layers[0].attn_norm;
    r.eps = hp.rms_eps;
    r.rows = nt;
    r.n = m->H;
    r.q16 = w.xa;
    r.ldq = (int64_t)m->nbH * 32;
    r.s16 = w.xa_s;
    r.ldqs = ntp;
    LAUNCH(kKRowQuant, row_quant_launch(r, st));
  }
  const int64_t kx = (int64_t)m->nbH * 32;
  const int64_t ntp_call = ((int64_t)nt + 127) / 128 * 128;  // captured scale planes' width
  for (int l = 0; l < hp.n_layer; ++l) {
    Layer& Ly = m->layers[l];
    const bool last = l == hp.n_layer - 1;
    // the last layer keeps all rows only through its K/V projections; after
    // that it carries the n_out tail rows: one row on the GEMV path, several
    // on the tensor-core path
    const bool tail1 = last && n_out == 1;
    const int r0 = last ? nt - n_out : 0;  // first row carried past attention
    const int mrows = nt - r0;
    const bool cap = dumps && l == m->dbg_layer;
    const bool cap_all = cap && !tail1;  // the tail rows: rows r0..nt-1 of the call
    int ns = 1, rc;
    if (cap) {
      for (auto& e : m->dbg)  // drop the previous call's captures
        if (e.second.first) cudaFree(e.second.first);
      m->dbg.clear();
      m->dbg_nt = nt;
      if ((rc = dbg_capture(m, st, "h_in", w.h, (size_t)nt * m->H * 4)) ||
          (rc = dbg_capture(m, st, "x_codes", w.xa, (size_t)nt * kx * 2)) ||
          (rc = dbg_capture_scales(m, st, "x_scales", w.xa_s, m->nbH, ntp, ntp_call)))
        return rc;
    }
    if ((rc = gemm_call(m, L, kKGemmQKV, xa, Ly.wqkv, nt, kEpiF32, true, w.part, m->qkvN, nullptr,
                        0, nullptr, 0, &ns)))
      return rc;
    AttnArgs at;
    at.q = w.qrot;
    at.qp[0] = w.qpl;
    at.qp[1] = w.qpl + (int64_t)w.max_nt * m->q;
    at.pos = pos;
    at.r0 = r0;
    at.r1 = nt;
    for (int i = 0; i < 4; ++i) at.shadow[i] = kv->plane(l, i);
    at.vt[0] = kv->vtp(l, 0);
    at.vt[1] = kv->vtp(l, 1);
    at.vt_ld = kv->vt_ld;
    at.nh = hp.n_head;
    at.nkv = hp.n_head_kv;
    at.hd = hp.head_dim;
    at.n_ctx = kv->n_ctx;
    at.nsplit = attention_nsplit(at.r1 - at.r0, at.nkv, m->num_sms, at.nh / at.nkv);
    if (tail1) row_attention_args(kv, l, &at);
    const bool attn_tc =
        attention_tc_supported(at) && attention_tc_preferred(at.r1 - at.r0, at.nh, m->num_sms);
    {
      RopeStoreArgs r;
      r.partials = w.part;
      r.nsplit = ns;
      r.split_stride = w.part_stride;
      r.bias = Ly.bqkv;
      r.pos = pos;
      r.nt = nt;
      r.nh = hp.n_head;
      r.nkv = hp.n_head_kv;
      r.hd = hp.head_dim;
      r.n_ctx = kv->n_ctx;
      r.cos_t = kv->cos_t;
      r.sin_t = kv->sin_t;
      // the rotated Q in f32 is read by the CUDA-core attention kernels and the
      // debug captures; the tensor-core attention reads only its fp16 hi/lo planes
      r.q_out = (attn_tc && !cap && !m->debug_f32) ? nullptr : w.qrot;
      r.q_planes[0] = w.qpl;
      r.q_planes[1] = w.qpl + (int64_t)w.max_nt * m->q;
      r.kreg = kv->k(l);
      r.vreg = kv->v(l);
      for (int i = 0; i < 4; ++i) r.shadow[i] = kv->plane(l, i);
      r.vt[0] = kv->vtp(l, 0);
      r.vt[1] = kv->vtp(l, 1);
      r.vt_ld = kv->vt_ld;
      r.status = m->d_status;
      if (hp.qk_norm) {
        r.q_norm = Ly.q_norm;
        r.k_norm = Ly.k_norm;
        r.eps = hp.rms_eps;
      }
      LAUNCH(kKRope, rope_store_launch(r, st));
    }
    if (cap) {
      auto& e = m->dbg["qkv"];
      const size_t bytes = (size_t)nt * m->qkvN * 4;
      if (e.second < bytes) {
        if (e.first) cudaFree(e.first);
        CK(cudaMalloc(&e.first, bytes));
        e.second = bytes;
      }
      CK(sum_splits_launch(w.part, ns, w.part_stride, (int64_t)nt * m->qkvN,
                           static_cast<float*>(e.first), st));
      if (cap_all && (rc = dbg_capture(m, st, "qrot", w.qrot, (size_t)nt * m->q * 4))) return rc;
    }
    AttnOut ao;
    ao.f32 = (m->debug_f32 || cap) ? w.att : nullptr;
    if (!tail1) {
      ao.q16 = w.xa;
      ao.ldq = (int64_t)m->nbq * 32;
      ao.s16 = w.xa_s;
      ao.ldqs = ntp;
      ao.row_base = r0;
    } else {
      ao.q8 = w.t_q;
      ao.s8 = w.t_s;
      ao.row_base = nt - 1;
    }
    if (attn_tc)
      LAUNCH(kKAttn, attention_tc_launch(at, ao, m->num_sms, m->d_status + 1, st));
    else
      LAUNCH(kKAttn, attention_launch(at, ao, st));
    if (cap_all) {
      if ((rc = dbg_capture(m, st, "att_codes", w.xa, (size_t)nt * m->nbq * 32 * 2)) ||
          (rc = dbg_capture_scales(m, st, "att_scales", w.xa_s, m->nbq, ntp, ntp_call)) ||
          (rc = dbg_capture(m, st, "att", w.att, (size_t)nt * m->q * 4)))
        return rc;
    }
    if (!tail1) {
      float* hr = w.h + (int64_t)r0 * m->H;  // the rows carried on
      GemmOperand xo_r = xo, xa_r = xa, xf_r = xf;
      xo_r.rows = xa_r.rows = xf_r.rows = mrows;
      if ((rc = gemm_call(m, L, kKGemmO, xo_r, Ly.wo, mrows, kEpiF32, true, w.part, m->H, nullptr,
                          0, nullptr, 0, &ns)))
        return rc;
      {
        RowQuantArgs r;
        r.h = hr;
        r.partials = w.part;
        r.nsplit = ns;
        r.split_stride = w.part_stride;
        r.norm_w = Ly.ffn_norm;
        r.eps = hp.rms_eps;
        r.rows = mrows;
        r.n = m->H;
        r.q16 = w.xa;
        r.ldq = (int64_t)m->nbH * 32;
        r.s16 = w.xa_s;
        r.ldqs = ntp;
        LAUNCH(kKRowQuant, row_quant_launch(r, st));
      }
      if (cap) {
        if ((rc = dbg_capture(m, st, "h_mid", w.h, (size_t)nt * m->H * 4)) ||
            (rc = dbg_capture(m, st, "f_codes", w.xa, (size_t)nt * kx * 2)) ||
            (rc = dbg_capture_scales(m, st, "f_scales", w.xa_s, m->nbH, ntp, ntp_call)))
          return rc;
      }
      float* s_f32 = nullptr;  // debug capture of the f32 values the SwiGLU epilogue quantizes
      if (cap) {
        auto& e = m->dbg["s_f32"];
        const size_t bytes = (size_t)nt * m->Fp * 4;
        if (e.second < bytes) {
          if (e.first) cudaFree(e.first);
          e.first = nullptr;
          e.second = 0;
          CK(cudaMalloc(&e.first, bytes));
          e.second = bytes;
        }
        CK(cudaMemsetAsync(e.first, 0, bytes, st));
        s_f32 = static_cast<float*>(e.first);  // rows as in "s_codes": the carried rows from 0
      }
      if ((rc = gemm_call(m, L, kKGemmGU, xa_r, Ly.wgu, mrows, kEpiSwiGLU, false, s_f32, m->Fp,
                          w.xf, m->Fp, w.xf_s, ntp, nullptr, l == m->fault_layer)))
        return rc;
      if (cap) {
        if ((rc = dbg_capture(m, st, "s_codes", w.xf, (size_t)nt * m->Fp * 2)) ||
            (rc = dbg_capture_scales(m, st, "s_scales", w.xf_s, m->nbF, ntp, ntp_call)))
          return rc;
      }
      if ((rc = gemm_call(m, L, kKGemmDown, xf_r, Ly.wd, mrows, kEpiF32, true, w.part, m->H,
                          nullptr, 0, nullptr, 0, &ns)))
        return rc;
      {
        RowQuantArgs r;
        r.h = hr;
        r.partials = w.part;
        r.nsplit = ns;
        r.split_stride = w.part_stride;
        r.norm_w = last ? m->out_norm : m->layers[l + 1].attn_norm;
        r.eps = hp.rms_eps;
        r.rows = mrows;
        r.n = m->H;
        r.q16 = w.xa;
        r.ldq = (int64_t)m->nbH * 32;
        r.s16 = w.xa_s;
        r.ldqs = ntp;
        LAUNCH(kKRowQuant, row_quant_launch(r, st));
      }
      if (dumps) dump_hidden(m, st, l + 1, hr, mrows);
      if (cap && (rc = dbg_capture(m, st, "h_out", w.h, (size_t)nt * m->H * 4))) return rc;
      if (last) {
        // lm_head over the n_out rows on the tensor cores, then one
        // status-gated copy into the caller's buffer
        if ((rc = gemm_call(m, L, kKLmHead, xa_r, m->lm_gemm, mrows, kEpiF32, false, w.lm_out,
                            m->V, nullptr, 0, nullptr, 0, nullptr)))
          return rc;
        LAUNCH(kKLmHead, copy_if_ok_launch(w.lm_out, logits, (int64_t)mrows * m->V, m->d_status, st));
      }
    } else {
      // last row only: o-projection, FFN, final norm, lm_head as GEMVs
      const int64_t last_row = nt - 1;
      // stage capture of the last row (debug): one-row layouts as in enqueue_decode
      auto cap_row = [&](const char* name, const void* src, size_t bytes) -> int {
        return cap ? dbg_capture(m, st, name, src, bytes) : MINFER_OK;
      };
      if ((rc = cap_row("att", w.att + last_row * m->q, (size_t)m->q * 4)) ||
          (rc = cap_row("att_q8", w.t_q, (size_t)m->nbq * 32)) ||
          (rc = cap_row("att_s8", w.t_s, (size_t)m->nbq * 4)))
        return rc;
      // o projection + residual of the last row, ffn_norm -> t_q/t_s
      if ((rc = row_gemv_norm(m, L,
                              row_gemv(m, Ly.wo_v, m->H, m->nbq, w.t_q, w.t_s, w.h_last,
                                       w.h + last_row * m->H),
                              Ly.ffn_norm, kTicketNormO, st)))
        return rc;
      if ((rc = cap_row("h_mid", w.h_last, (size_t)m->H * 4)) ||
          (rc = cap_row("f_q8", w.t_q, (size_t)m->nbH * 32)) ||
          (rc = cap_row("f_s8", w.t_s, (size_t)m->nbH * 4)))
        return rc;
      // gate/up + SwiGLU -> t_q2/t_s2
      if ((rc = row_gemv_swiglu(m, L, Ly.wgu_v, st))) return rc;
      if ((rc = cap_row("s_q8", w.t_q2, (size_t)m->nbF * 32)) ||
          (rc = cap_row("s_s8", w.t_s2, (size_t)m->nbF * 4)))
        return rc;
      // down + residual, output norm -> t_q/t_s
      if ((rc = row_gemv_norm(m, L,
                              row_gemv(m, Ly.wd_v, m->H, m->nbF, w.t_q2, w.t_s2, w.h_last, w.h_last),
                              m->out_norm, kTicketNormDown, st)))
        return rc;
      if ((rc = cap_row("h_out", w.h_last, (size_t)m->H * 4))) return rc;
      if (dumps) dump_hidden(m, st, l + 1, w.h_last, 1);
      {
        const GemvW& out = hp.tied_embeddings ? m->tok_embd : m->output;
        GemvArgs g = row_gemv(m, out, m->V, m->nbH, w.t_q, w.t_s, logits, nullptr);
        g.status = m->d_status;
        LAUNCH(kKLmHead, gemv_launch(g, st));
      }
    }
  }
  return MINFER_OK;
}

// Run (record or replay) the forward on stream st.
// The lm_head in the tensor-core layout, and the workspace for n_out logits
// rows (both only when a call asks for more than one row).
int ensure_logits(minfer_model* m, int n_out) {
  Workspace& w = m->ws;
  if (n_out <= 1) return MINFER_OK;
  int rc;
  if (!m->lm_gemm.codes) {
    const GemvW& src = m->hp.tied_embeddings ? m->tok_embd : m->output;
    if ((rc = m->lm_gemm.alloc(m->V, m->nbH))) return rc;
    CK(gemv_to_gemm_launch(src.q, src.s, m->V, m->nbH, m->lm_gemm.codes, m->lm_gemm.scales,
                           m->lm_gemm.rows_pad, m->stream));
    CK(cudaStreamSynchronize(m->stream));
  }
  if (n_out <= w.logits_rows) return MINFER_OK;
  if (m->gexec) {
    cudaGraphExecDestroy(m->gexec);
    m->gexec = nullptr;
  }
  if (m->graph) {
    cudaGraphDestroy(m->graph);
    m->graph = nullptr;
  }
  dfree(w.logits);
  dfree(w.lm_out);
  w.logits_rows = 0;
  if ((rc = dalloc(&w.logits, (size_t)n_out * m->V)) || (rc = dalloc(&w.lm_out, (size_t)n_out * m->V)))
    return rc;
  w.logits_rows = n_out;
  return MINFER_OK;
}

int run_forward(minfer_model* m, minfer_kv* kv, const int32_t* ids, const int32_t* pos, int nt,
                int n_out, float* logits, cudaStream_t st) {
  int rc = ensure_workspace(m, nt);
  if (rc) return rc;
  if ((rc = ensure_logits(m, n_out))) return rc;
  m->dump_on = m->dump_host != nullptr && nt <= m->dump_max_nt;
  const bool dumps = m->dump_on || m->dbg_layer >= 0 || m->fault_layer >= 0;
  if (dumps) {
    // dumps copy to host memory mid-sequence: run eagerly
    m->ev_used = 0;
    rc = enqueue_forward(m, kv, ids, pos, nt, n_out, logits, st, m->profile, true);
    return rc;
  }
  minfer_model::GraphKey key;
  key.nt = nt;
  key.n_out = n_out;
  key.kv = kv;
  key.ids = ids;
  key.pos = pos;
  key.logits = logits;
  key.profile = m->profile;
  if (!m->gexec || !(key == m->gkey)) {
    if (m->gexec) {
      cudaGraphExecDestroy(m->gexec);
      m->gexec = nullptr;
    }
    if (m->graph) {
      cudaGraphDestroy(m->graph);
      m->graph = nullptr;
    }
    m->ev_used = 0;
    CK(cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal));
    rc = enqueue_forward(m, kv, ids, pos, nt, n_out, logits, st, m->profile, false);
    cudaGraph_t g = nullptr;
    cudaError_t e = cudaStreamEndCapture(st, &g);
    if (rc) {
      if (g) cudaGraphDestroy(g);
      return rc;
    }
    CK(e);
    m->graph = g;
    CK(cudaGraphInstantiate(&m->gexec, g, 0));
    m->gkey = key;
  }
  CK(cudaGraphLaunch(m->gexec, st));
  return MINFER_OK;
}

int finish_status(minfer_model* m, cudaStream_t st) {
  CK(cudaMemcpyAsync(m->h_status, m->d_status, 2 * sizeof(int), cudaMemcpyDeviceToHost, st));
  CK(cudaStreamSynchronize(st));
  if (m->profile) {
    for (int i = 0; i + 1 < m->ev_used; i += 2) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, m->ev[i], m->ev[i + 1]) == cudaSuccess) {
        m->prof_ms[m->ev_class[i]] += ms;
        m->prof_n[m->ev_class[i]] += 1;
      }
    }
    (void)cudaGetLastError();  // a failed timing query must not leak into the next launch check
  }
  if (m->h_status[1] != 0) {
    m->last_device_status = m->h_status[1];
    snprintf(g_last_error, sizeof g_last_error, "device wait timed out (code %d)", m->h_status[1]);
    return MINFER_ERR_DEVICE;
  }
  return m->h_status[0];
}

void rope_tables(int n_ctx, int hd, float theta, std::vector<float>& c, std::vector<float>& s) {
  // cos/sin of p * theta^(-2i/hd), evaluated in double and rounded to f32
  const int half = hd / 2;
  c.assign((size_t)n_ctx * half, 0.f);
  s.assign((size_t)n_ctx * half, 0.f);
  for (int i = 0; i < half; ++i) {
    const double f = std::pow((double)theta, -2.0 * (double)i / (double)hd);
    for (int p = 0; p < n_ctx; ++p) {
      const double ang = (double)p * f;
      c[(size_t)p * half + i] = (float)std::cos(ang);
      s[(size_t)p * half + i] = (float)std::sin(ang);
    }
  }
}

int check_device(const minfer_model* m) {
  int dev = -1;
  CK(cudaGetDevice(&dev));
  if (dev != m->device) return MINFER_ERR_STATE;
  return MINFER_OK;
}

}  // namespace

// ====================================================================== C ABI

extern "C" {

int minfer_model_create(const minfer_hparams* hp, minfer_model** out) {
  if (!hp || !out) return MINFER_ERR_ARG;
  *out = nullptr;
  if (hp->n_layer <= 0 || hp->n_embd <= 0 || hp->n_head <= 0 || hp->n_head_kv <= 0 ||
      hp->n_head % hp->n_head_kv != 0 || hp->head_dim <= 0 || hp->n_ff <= 0 || hp->n_vocab <= 0 ||
      hp->max_seq_len <= 0)
    return MINFER_ERR_ARG;
  if (!(hp->head_dim == 64 || hp->head_dim == 128) || hp->n_head / hp->n_head_kv > 8 ||
      hp->n_embd > 4096 || (int64_t)hp->n_head * hp->head_dim > 4096)
    return MINFER_ERR_SHAPE;
  minfer_model* m = new minfer_model();
  m->hp = *hp;
  cudaError_t e = cudaGetDevice(&m->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&m->stream, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    record_cuda_error(e, "model_create", __LINE__);
    delete m;
    return MINFER_ERR_CUDA;
  }
  int rc = model_alloc(m);
  if (rc) {
    model_release(m);
    delete m;
    return rc;
  }
  *out = m;
  return MINFER_OK;
}

int minfer_model_set_tensor(minfer_model* m, const minfer_tensor* t) {
  if (!m) return MINFER_ERR_ARG;
  int rc = check_device(m);
  if (rc) return rc;
  return set_tensor(m, t);
}

int minfer_model_finalize(minfer_model* m) {
  if (!m) return MINFER_ERR_ARG;
  for (const auto& n : required_names(m->hp))
    if (!m->have.count(n)) {
      snprintf(g_last_error, sizeof g_last_error, "missing tensor %s", n.c_str());
      return MINFER_ERR_MISSING_TENSOR;
    }
  // staging buffers are not needed after load
  if (m->stage) cudaFree(m->stage);
  m->stage = nullptr;
  m->stage_bytes = 0;
  dfree(m->stage_q);
  dfree(m->stage_d);
  m->stage_q_bytes = 0;
  m->finalized = true;
  return MINFER_OK;
}

int minfer_load_weights(const minfer_hparams* hp, const minfer_tensor* tensors, int n,
                        minfer_model** out) {
  if (!out || (n > 0 && !tensors)) return MINFER_ERR_ARG;
  minfer_model* m = nullptr;
  int rc = minfer_model_create(hp, &m);
  if (rc) return rc;
  for (int i = 0; i < n && !rc; ++i) rc = set_tensor(m, &tensors[i]);
  if (!rc) rc = minfer_model_finalize(m);
  if (rc) {
    minfer_free(m);
    return rc;
  }
  *out = m;
  return MINFER_OK;
}

void minfer_free(minfer_model* m) {
  if (!m) return;
  cudaDeviceSynchronize();
  model_release(m);
  delete m;
}

int minfer_kv_create(minfer_model* m, int n_ctx, minfer_kv** out) {
  if (!m || !out || n_ctx <= 0) return MINFER_ERR_ARG;
  *out = nullptr;
  int rc = check_device(m);
  if (rc) return rc;
  minfer_kv* kv = new minfer_kv();
  kv->m = m;
  kv->n_ctx = std::min(n_ctx, m->hp.max_seq_len);
  kv->vt_ld = rup(kv->n_ctx, 64);
  kv->m_kvw = m->kvw;
  std::vector<float> c, s;
  rope_tables(kv->n_ctx, m->hp.head_dim, m->hp.rope_theta, c, s);
  if ((rc = dalloc(&kv->regions, (size_t)m->hp.n_layer * 2 * kv->n_ctx * m->kvw)) ||
      (rc = dalloc(&kv->shadow, (size_t)m->hp.n_layer * 4 * kv->n_ctx * m->kvw)) ||
      (rc = dalloc(&kv->vt, (size_t)m->hp.n_layer * 2 * m->kvw * kv->vt_ld)) ||
      (rc = dalloc(&kv->cos_t, c.size())) || (rc = dalloc(&kv->sin_t, s.size())) ||
      (rc = dalloc(&kv->seen, (size_t)(kv->n_ctx + 31) / 32))) {
    minfer_kv_free(kv);
    return rc;
  }
  if (cudaMemcpy(kv->cos_t, c.data(), c.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(kv->sin_t, s.data(), s.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess) {
    minfer_kv_free(kv);
    return MINFER_ERR_CUDA;
  }
  *out = kv;
  return MINFER_OK;
}

int minfer_kv_n_ctx(const minfer_kv* kv) { return kv ? kv->n_ctx : 0; }

void minfer_kv_free(minfer_kv* kv) {
  if (!kv) return;
  cudaDeviceSynchronize();
  if (kv->m && kv->m->gkey.kv == kv && kv->m->gexec) {
    cudaGraphExecDestroy(kv->m->gexec);
    kv->m->gexec = nullptr;
    if (kv->m->graph) cudaGraphDestroy(kv->m->graph);
    kv->m->graph = nullptr;
    kv->m->gkey = minfer_model::GraphKey();
  }
  dfree(kv->regions);
  dfree(kv->shadow);
  dfree(kv->vt);
  dfree(kv->cos_t);
  dfree(kv->sin_t);
  dfree(kv->seen);
  delete kv;
}

int minfer_kv_read(const minfer_kv* kv, int layer, int which, int row0, int nrows, float* out) {
  if (!kv || !out || layer < 0 || layer >= kv->m->hp.n_layer || (which != 0 && which != 1) ||
      row0 < 0 || nrows < 0 || row0 + nrows > kv->n_ctx)
    return MINFER_ERR_ARG;
  const float* src = (which ? kv->v(layer) : kv->k(layer)) + (int64_t)row0 * kv->m->kvw;
  CK(cudaDeviceSynchronize());
  CK(cudaMemcpy(out, src, (size_t)nrows * kv->m->kvw * 4, cudaMemcpyDeviceToHost));
  return MINFER_OK;
}

int minfer_kv_write(minfer_kv* kv, int layer, int which, int row0, int nrows, const float* in) {
  if (!kv || !in || layer < 0 || layer >= kv->m->hp.n_layer || (which != 0 && which != 1) ||
      row0 < 0 || nrows < 0 || row0 + nrows > kv->n_ctx)
    return MINFER_ERR_ARG;
  float* dst = (which ? kv->v(layer) : kv->k(layer)) + (int64_t)row0 * kv->m->kvw;
  CK(cudaDeviceSynchronize());
  CK(cudaMemcpy(dst, in, (size_t)nrows * kv->m->kvw * 4, cudaMemcpyHostToDevice));
  // keep the fp16 hi/lo copies the attention reads in step with the regions
  const int64_t off = (int64_t)row0 * kv->m->kvw;
  __half* planes[4];
  for (int i = 0; i < 4; ++i) planes[i] = kv->plane(layer, i) + off;
  __half* vt[2] = {kv->vtp(layer, 0), kv->vtp(layer, 1)};
  CK(kv_shadow_launch(kv->k(layer) + off, kv->v(layer) + off, (int64_t)nrows * kv->m->kvw, planes,
                      vt, kv->vt_ld, row0, (int)kv->m->kvw, 0));
  CK(cudaDeviceSynchronize());
  return MINFER_OK;
}

int minfer_prefill(minfer_model* m, const int32_t* token_ids, const int32_t* positions,
                   int n_tokens, minfer_kv* kv, float* logits_out) {
  return minfer_prefill_n(m, token_ids, positions, n_tokens, kv, 1, logits_out);
}

int minfer_prefill_n(minfer_model* m, const int32_t* token_ids, const int32_t* positions,
                     int n_tokens, minfer_kv* kv, int n_out, float* logits_out) {
  if (!m || !token_ids || !positions || !kv || !logits_out || n_tokens <= 0 || kv->m != m ||
      n_out < 1 || n_out > n_tokens)
    return MINFER_ERR_ARG;
  if (!m->finalized) return MINFER_ERR_STATE;
  int rc = check_device(m);
  if (rc) return rc;
  // host preflight: nothing is written when it fails
  std::vector<uint8_t> seen((size_t)kv->n_ctx, 0);
  for (int t = 0; t < n_tokens; ++t) {
    const int p = positions[t];
    if (p < 0 || p >= kv->n_ctx) return MINFER_ERR_POS_OOB;
  }
  for (int t = 0; t < n_tokens; ++t)
    if (token_ids[t] < 0 || token_ids[t] >= m->hp.n_vocab) return MINFER_ERR_TOKEN_OOB;
  for (int t = 0; t < n_tokens; ++t) {
    if (seen[positions[t]]) return MINFER_ERR_ARG;
    seen[positions[t]] = 1;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if ((rc = ensure_workspace(m, n_tokens))) return rc;
  cudaStream_t st = m->stream;
  CK(cudaMemcpyAsync(m->ws.ids, token_ids, (size_t)n_tokens * 4, cudaMemcpyHostToDevice, st));
  CK(cudaMemcpyAsync(m->ws.pos, positions, (size_t)n_tokens * 4, cudaMemcpyHostToDevice, st));
  if ((rc = ensure_logits(m, n_out))) return rc;
  if ((rc = run_forward(m, kv, m->ws.ids, m->ws.pos, n_tokens, n_out, m->ws.logits, st))) return rc;
  // the caller's buffer is written only when the call succeeded
  if ((rc = finish_status(m, st))) return rc;
  CK(cudaMemcpyAsync(logits_out, m->ws.logits, (size_t)n_out * m->V * 4, cudaMemcpyDeviceToHost,
                     st));
  CK(cudaStreamSynchronize(st));
  return MINFER_OK;
}

int minfer_prefill_device(minfer_model* m, const int32_t* d_token_ids, const int32_t* d_positions,
                          int n_tokens, minfer_kv* kv, float* d_logits, void* stream) {
  return minfer_prefill_device_n(m, d_token_ids, d_positions, n_tokens, kv, 1, d_logits, stream);
}

int minfer_prefill_device_n(minfer_model* m, const int32_t* d_token_ids,
                            const int32_t* d_positions, int n_tokens, minfer_kv* kv, int n_out,
                            float* d_logits, void* stream) {
  if (!m || !d_token_ids || !d_positions || !kv || !d_logits || n_tokens <= 0 || kv->m != m ||
      n_out < 1 || n_out > n_tokens)
    return MINFER_ERR_ARG;
  if (!m->finalized) return MINFER_ERR_STATE;
  int rc = check_device(m);
  if (rc) return rc;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaStream_t st = stream ? static_cast<cudaStream_t>(stream) : m->stream;
  return run_forward(m, kv, d_token_ids, d_positions, n_tokens, n_out, d_logits, st);
}

int minfer_sync_status(minfer_model* m, void* stream) {
  if (!m) return MINFER_ERR_ARG;
  cudaStream_t st = stream ? static_cast<cudaStream_t>(stream) : m->stream;
  return finish_status(m, st);
}

int minfer_set_dump(minfer_model* m, float* host_hidden, int max_tokens) {
  if (!m || (host_hidden && max_tokens <= 0)) return MINFER_ERR_ARG;
  m->dump_host = host_hidden;
  m->dump_max_nt = host_hidden ? max_tokens : 0;
  m->debug_f32 = host_hidden != nullptr;
  return MINFER_OK;
}

int minfer_profile_enable(minfer_model* m, int enable) {
  if (!m) return MINFER_ERR_ARG;
  m->profile = enable != 0;
  for (int k = 0; k < kNumKClass; ++k) {
    m->prof_ms[k] = 0.0;
    m->prof_n[k] = 0;
  }
  return MINFER_OK;
}

int minfer_profile_read(minfer_model* m, int k, const char** name, int64_t* launches,
                        double* total_ms) {
  if (!m || k < 0 || k >= kNumKClass) return MINFER_ERR_ARG;
  if (name) *name = kClassNames[k];
  if (launches) *launches = m->prof_n[k];
  if (total_ms) *total_ms = m->prof_ms[k];
  return MINFER_OK;
}

// ---------------------------------------------------------------- single stages

int minfer_op_quantize(const float* d_x, int64_t rows, int64_t n, int8_t* d_q, uint16_t* d_d) {
  if (!d_x || !d_q || !d_d || rows <= 0 || n <= 0 || n > 4096) return MINFER_ERR_ARG;
  RowQuantArgs r;
  r.h = const_cast<float*>(d_x);
  r.rows = rows;
  r.n = n;
  r.q8 = d_q;
  float* s = nullptr;
  int rc = dalloc(&s, (size_t)rows * ((n + 31) / 32));
  if (rc) return rc;
  r.s8 = s;
  r.s8_bits = d_d;
  cudaError_t e = row_quant_launch(r, 0);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  dfree(s);
  CK(e);
  return MINFER_OK;
}

int minfer_op_rmsnorm_quantize(const float* d_x, const float* d_w, int64_t rows, int64_t n,
                               float eps, int8_t* d_q, uint16_t* d_d) {
  if (!d_x || !d_w || !d_q || !d_d || rows <= 0 || n <= 0 || n > 4096) return MINFER_ERR_ARG;
  RowQuantArgs r;
  r.h = const_cast<float*>(d_x);
  r.norm_w = d_w;
  r.eps = eps;
  r.rows = rows;
  r.n = n;
  r.q8 = d_q;
  float* s = nullptr;
  int rc = dalloc(&s, (size_t)rows * ((n + 31) / 32));
  if (rc) return rc;
  r.s8 = s;
  r.s8_bits = d_d;
  cudaError_t e = row_quant_launch(r, 0);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  dfree(s);
  CK(e);
  return MINFER_OK;
}

namespace {
// Canonical int8 + fp16 bits -> GEMM planes (test helper).
int planes_from_q8(const int8_t* q, const uint16_t* d, int64_t rows, int nb, GemmW& w,
                   int interleave, int which, bool alloc) {
  int rc;
  if (alloc && (rc = w.alloc(interleave ? 2 * rup(rows, 32) : rows, nb))) return rc;
  RepackArgs r;
  r.q = q;
  r.dbits = d;
  r.rows = rows;
  r.nb = nb;
  r.dst_codes = w.codes;
  r.dst_scales = w.scales;
  r.dst_rows_pad = w.rows_pad;
  r.interleave = interleave;
  r.which = which;
  CK(repack_gemm_launch(r, 0));
  return MINFER_OK;
}
}  // namespace

int minfer_op_gemm(const int8_t* d_xq, const uint16_t* d_xd, int64_t M, const int8_t* d_wq,
                   const uint16_t* d_wd, int64_t N, int64_t K, float* d_y, int32_t* d_dots) {
  if (!d_xq || !d_xd || !d_wq || !d_wd || !d_y || M <= 0 || N <= 0 || K <= 0) return MINFER_ERR_ARG;
  const int nb = (int)((K + 31) / 32);
  int num_sms = 148, dev = 0;
  CK(cudaGetDevice(&dev));
  CK(cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev));
  GemmW A, B;
  float* part = nullptr;
  int rc = planes_from_q8(d_xq, d_xd, M, nb, A, 0, 0, true);
  if (!rc) rc = planes_from_q8(d_wq, d_wd, N, nb, B, 0, 0, true);
  GemmLaunch g;
  g.A = A.op();
  g.B = B.op();
  g.M = M;
  g.N = N;
  g.epi = d_dots ? kEpiDots : kEpiF32;
  g.plan = gemm_plan(M, N, nb, num_sms, d_dots == nullptr);
  g.plan.splits = std::min(g.plan.splits, kMaxSplits);
  const int stages = (nb + 1) / 2;
  int splits = std::max(1, std::min(g.plan.splits, stages));
  const int sps = (stages + splits - 1) / splits;
  splits = (stages + sps - 1) / sps;
  if (!rc) rc = dalloc(&part, (size_t)splits * M * N);
  int* err = nullptr;
  if (!rc) rc = dalloc(&err, 1);
  g.out = part;
  g.ldo = N;
  g.split_stride = M * N;
  g.dots = d_dots;
  g.err = err;
  GemmMaps maps;
  if (!rc && gemm_make_maps(g.A, g.B, g.plan.bn, &maps)) rc = MINFER_ERR_CUDA;
  cudaError_t e = cudaSuccess;
  if (!rc) e = gemm_launch(g, maps, num_sms, 0);
  if (!rc && e == cudaSuccess) e = sum_splits_launch(part, splits, M * N, M * N, d_y, 0);
  if (!rc && e == cudaSuccess) e = cudaDeviceSynchronize();
  int herr = 0;
  if (!rc && e == cudaSuccess) cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost);
  A.release();
  B.release();
  dfree(part);
  dfree(err);
  if (rc) return rc;
  CK(e);
  return herr ? MINFER_ERR_DEVICE : MINFER_OK;
}

int minfer_op_gemm_swiglu(const int8_t* d_xq, const uint16_t* d_xd, int64_t M, const int8_t* d_gq,
                          const uint16_t* d_gd, const int8_t* d_uq, const uint16_t* d_ud, int64_t F,
                          int64_t K, int8_t* d_sq, uint16_t* d_sd) {
  if (!d_xq || !d_xd || !d_gq || !d_gd || !d_uq || !d_ud || !d_sq || !d_sd || M <= 0 || F <= 0 ||
      K <= 0)
    return MINFER_ERR_ARG;
  const int nb = (int)((K + 31) / 32);
  const int nbF = (int)((F + 31) / 32);
  const int64_t Fp = (int64_t)nbF * 32;
  int num_sms = 148, dev = 0;
  CK(cudaGetDevice(&dev));
  CK(cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev));
  GemmW A, B;
  int rc = planes_from_q8(d_xq, d_xd, M, nb, A, 0, 0, true);
  if (!rc) rc = B.alloc(2 * Fp, nb);
  if (!rc) rc = planes_from_q8(d_gq, d_gd, F, nb, B, 1, 0, false);
  if (!rc) rc = planes_from_q8(d_uq, d_ud, F, nb, B, 1, 1, false);
  const int64_t Mp = rup(M, 128);
  __half* codes = nullptr;
  float* scales = nullptr;
  int* err = nullptr;
  if (!rc) rc = dalloc(&codes, (size_t)M * Fp);
  if (!rc) rc = dalloc(&scales, (size_t)nbF * Mp);
  if (!rc) rc = dalloc(&err, 1);
  GemmLaunch g;
  g.A = A.op();
  g.B = B.op();
  g.M = M;
  g.N = 2 * Fp;
  g.epi = kEpiSwiGLU;
  g.plan = gemm_plan(M, 2 * Fp, nb, num_sms, false);
  g.q_out = codes;
  g.ldq = Fp;
  g.qs_out = scales;
  g.ldqs = Mp;
  g.n_out_cols = Fp;
  g.err = err;
  GemmMaps maps;
  if (!rc && gemm_make_maps(g.A, g.B, g.plan.bn, &maps)) rc = MINFER_ERR_CUDA;
  cudaError_t e = cudaSuccess;
  if (!rc) e = gemm_launch(g, maps, num_sms, 0);
  if (!rc && e == cudaSuccess) e = gemm_plane_to_q8_launch(codes, scales, M, Mp, nbF, d_sq, d_sd, 0);
  if (!rc && e == cudaSuccess) e = cudaDeviceSynchronize();
  int herr = 0;
  if (!rc && e == cudaSuccess) cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost);
  A.release();
  B.release();
  dfree(codes);
  dfree(scales);
  dfree(err);
  if (rc) return rc;
  CK(e);
  return herr ? MINFER_ERR_DEVICE : MINFER_OK;
}

int minfer_op_attention(const float* d_q, const int32_t* d_pos, int nt, const float* d_k,
                        const float* d_v, int n_ctx, int n_head, int n_head_kv, int head_dim,
                        float* d_o) {
  if (!d_q || !d_pos || !d_k || !d_v || !d_o || nt <= 0 || n_ctx <= 0 || n_head_kv <= 0 ||
      n_head % n_head_kv != 0 || head_dim % 32 != 0)
    return MINFER_ERR_ARG;
  int num_sms = 148, dev = 0;
  CK(cudaGetDevice(&dev));
  CK(cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev));
  const int64_t kvw = (int64_t)n_head_kv * head_dim;
  const int64_t q = (int64_t)n_head * head_dim;
  AttnArgs a;
  a.q = d_q;
  a.pos = d_pos;
  a.r0 = 0;
  a.r1 = nt;
  a.nh = n_head;
  a.nkv = n_head_kv;
  a.hd = head_dim;
  a.n_ctx = n_ctx;
  a.nsplit = attention_nsplit(nt, n_head_kv, num_sms, n_head / n_head_kv);
  __half* sh = nullptr;
  float* s16 = nullptr;
  __half* q16 = nullptr;
  const int64_t vt_ld = rup(n_ctx, 64);
  __half* vt = nullptr;
  __half* qpl = nullptr;
  int rc = dalloc(&sh, (size_t)4 * n_ctx * kvw);
  if (!rc) rc = dalloc(&vt, (size_t)2 * kvw * vt_ld);
  if (!rc) rc = dalloc(&qpl, (size_t)2 * nt * q);
  if (!rc) rc = dalloc(&q16, (size_t)nt * q);
  if (!rc) rc = dalloc(&s16, (size_t)(q / 32) * nt);
  // one query row: the cluster kernel, straight from the f32 regions
  if (nt == 1) {
    a.kreg = d_k;
    a.vreg = d_v;
  }
  cudaError_t e = cudaSuccess;
  if (!rc) {
    __half* planes[4];
    for (int i = 0; i < 4; ++i) {
      planes[i] = sh + (int64_t)i * n_ctx * kvw;
      a.shadow[i] = planes[i];
    }
    __half* vtp[2] = {vt, vt + kvw * vt_ld};
    a.vt[0] = vtp[0];
    a.vt[1] = vtp[1];
    a.vt_ld = vt_ld;
    AttnOut out;
    out.q16 = q16;
    out.ldq = q;
    out.s16 = s16;
    out.ldqs = nt;
    out.f32 = d_o;
    a.qp[0] = qpl;
    a.qp[1] = qpl + (int64_t)nt * q;
    e = kv_shadow_launch(d_k, d_v, (int64_t)n_ctx * kvw, planes, vtp, vt_ld, 0, (int)kvw, 0);
    if (e == cudaSuccess) e = split_planes_launch(d_q, (int64_t)nt * q, qpl, qpl + (int64_t)nt * q, 0);
    int* err = nullptr;
    if (dalloc(&err, 1) != MINFER_OK) e = cudaErrorMemoryAllocation;
    if (e == cudaSuccess)
      e = attention_tc_supported(a) ? attention_tc_launch(a, out, num_sms, err, 0)
                                    : attention_launch(a, out, 0);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    int herr = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&herr, err, sizeof(int), cudaMemcpyDeviceToHost);
    dfree(err);
    if (e == cudaSuccess && herr != 0) {
      snprintf(g_last_error, sizeof g_last_error, "device wait timed out (code %d)", herr);
      e = cudaErrorLaunchTimeout;
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
  }
  dfree(sh);
  dfree(vt);
  dfree(qpl);
  dfree(q16);
  dfree(s16);
  if (rc) return rc;
  CK(e);
  return MINFER_OK;
}

int minfer_op_rope_store(const float* d_qkv, const float* d_bias, const int32_t* d_pos, int nt,
                         int n_head, int n_head_kv, int head_dim, float theta, int n_ctx,
                         float* d_q_out, float* d_k, float* d_v) {
  return minfer_op_qknorm_rope_store(d_qkv, d_bias, nullptr, nullptr, 0.f, d_pos, nt, n_head,
                                     n_head_kv, head_dim, theta, n_ctx, d_q_out, d_k, d_v);
}

int minfer_op_qknorm_rope_store(const float* d_qkv, const float* d_bias, const float* d_qnorm,
                                const float* d_knorm, float eps, const int32_t* d_pos, int nt,
                                int n_head, int n_head_kv, int head_dim, float theta, int n_ctx,
                                float* d_q_out, float* d_k, float* d_v) {
  if (!d_qkv || !d_pos || !d_q_out || !d_k || !d_v || nt <= 0 || n_ctx <= 0) return MINFER_ERR_ARG;
  if ((d_qnorm == nullptr) != (d_knorm == nullptr)) return MINFER_ERR_ARG;
  std::vector<float> c, s;
  rope_tables(n_ctx, head_dim, theta, c, s);
  float *dc = nullptr, *ds = nullptr;
  int rc = dalloc(&dc, c.size());
  if (!rc) rc = dalloc(&ds, s.size());
  cudaError_t e = cudaSuccess;
  if (!rc) e = cudaMemcpy(dc, c.data(), c.size() * 4, cudaMemcpyHostToDevice);
  if (!rc && e == cudaSuccess) e = cudaMemcpy(ds, s.data(), s.size() * 4, cudaMemcpyHostToDevice);
  RopeStoreArgs a;
  a.partials = d_qkv;
  a.nsplit = 1;
  a.bias = d_bias;
  a.pos = d_pos;
  a.nt = nt;
  a.nh = n_head;
  a.nkv = n_head_kv;
  a.hd = head_dim;
  a.n_ctx = n_ctx;
  a.cos_t = dc;
  a.sin_t = ds;
  a.q_out = d_q_out;
  a.kreg = d_k;
  a.vreg = d_v;
  a.q_norm = d_qnorm;
  a.k_norm = d_knorm;
  a.eps = eps;
  __half* sh = nullptr;
  const int64_t kvw = (int64_t)n_head_kv * head_dim;
  const int64_t vt_ld = rup(n_ctx, 64);
  __half* vt = nullptr;
  if (!rc) rc = dalloc(&sh, (size_t)4 * n_ctx * kvw);
  if (!rc) rc = dalloc(&vt, (size_t)2 * kvw * vt_ld);
  if (!rc) {
    for (int i = 0; i < 4; ++i) a.shadow[i] = sh + (int64_t)i * n_ctx * kvw;
    a.vt[0] = vt;
    a.vt[1] = vt + kvw * vt_ld;
    a.vt_ld = vt_ld;
  }
  if (!rc && e == cudaSuccess) e = rope_store_launch(a, 0);
  if (!rc && e == cudaSuccess) e = cudaDeviceSynchronize();
  dfree(dc);
  dfree(ds);
  dfree(sh);
  dfree(vt);
  if (rc) return rc;
  CK(e);
  return MINFER_OK;
}

int minfer_debug_layer(minfer_model* m, int layer) {
  if (!m || layer < -1 || layer >= m->hp.n_layer) return MINFER_ERR_ARG;
  m->dbg_layer = layer;
  return MINFER_OK;
}

int minfer_debug_read(minfer_model* m, const char* buffer, void* host, int64_t bytes) {
  if (!m || !buffer || !host) return MINFER_ERR_ARG;
  {
    auto it = m->dbg.find(buffer);
    if (it != m->dbg.end() && it->second.first) {
      if (bytes < (int64_t)it->second.second) return MINFER_ERR_ARG;
      CK(cudaDeviceSynchronize());
      CK(cudaMemcpy(host, it->second.first, it->second.second, cudaMemcpyDeviceToHost));
      return MINFER_OK;
    }
  }
  if (m->ws.max_nt == 0) return MINFER_ERR_ARG;
  const Workspace& w = m->ws;
  const std::string b(buffer);
  const void* src = nullptr;
  int64_t n = 0;
  if (b == "h") { src = w.h; n = (int64_t)w.max_nt * m->H * 4; }
  else if (b == "att") { src = w.att; n = (int64_t)w.max_nt * m->q * 4; }
  else if (b == "xf") { src = w.xf; n = (int64_t)w.max_nt * m->Fp * 2; }
  else if (b == "xf_s") { src = w.xf_s; n = (int64_t)m->nbF * w.ntp * 4; }
  else return MINFER_ERR_ARG;
  if (bytes < n) return MINFER_ERR_ARG;
  CK(cudaDeviceSynchronize());
  CK(cudaMemcpy(host, src, (size_t)n, cudaMemcpyDeviceToHost));
  return MINFER_OK;
}

const char* minfer_strerror(int code) {
  switch (code) {
    case MINFER_OK: return "ok";
    case MINFER_ERR_ARG: return "invalid argument";
    case MINFER_ERR_POS_OOB: return "position out of range of the KV regions";
    case MINFER_ERR_TOKEN_OOB: return "token id out of range of the vocabulary";
    case MINFER_ERR_MISSING_TENSOR: return "missing tensor";
    case MINFER_ERR_SHAPE: return "unknown tensor or wrong shape/type";
    case MINFER_ERR_CUDA: return g_last_error[0] ? g_last_error : "CUDA error";
    case MINFER_ERR_OOM: return "device out of memory";
    case MINFER_ERR_DEVICE: return "device-side wait timed out";
    case MINFER_ERR_STATE: return "call order or device violated";
    case MINFER_ERR_TOO_LARGE: return "problem larger than the fixed scratch area";
    default: return "unknown error";
  }
}

int minfer_device_status(minfer_model* m) { return m ? m->last_device_status : 0; }

int minfer_debug_fault(minfer_model* m, int layer, int64_t wait_limit_ns) {
  if (!m || layer < -1 || layer >= m->hp.n_layer || (layer >= 0 && wait_limit_ns <= 0))
    return MINFER_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  m->fault_layer = layer;
  m->fault_wait_ns = layer >= 0 ? (uint64_t)wait_limit_ns : 0;
  return MINFER_OK;
}

}  // extern "C"
