// kernels.h -- host-side launchers of the sm_103a kernels (one translation
// unit per kernel family) and the device data layouts they share.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace minfer {

// Launch with programmatic stream serialization (see pdl_trigger/pdl_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- layouts
//
// GEMM operand planes (tensor-core path):
//   codes  fp16 [rows][kpad]   integer values -127..127 held exactly in fp16,
//                              kpad = nb * 32, zero beyond the real columns
//   scales f32  [nb][rows_pad] f32 value of each block's fp16 scale, stored
//                              block-major ("transposed") so a tile's scales
//                              are one contiguous box per block
// GEMV planes (one-row tail):
//   codes  int8 [rows][kpad], scales f32 [rows][nb]

struct GemmOperand {
  const __half* codes = nullptr;  // [rows][kpad]
  const float* scales = nullptr;  // [nb][rows_pad]
  int64_t rows = 0, rows_pad = 0;
  int nb = 0;
};

// Gate/up weights for the SwiGLU epilogue: rows interleaved in groups of
// kSwiGluGroup gate rows then the kSwiGluGroup up rows of the same outputs,
// so that one epilogue warp's 64 columns hold matching gate and up values.
constexpr int kSwiGluGroup = 32;

enum GemmEpilogue : int {
  kEpiF32 = 0,     // out[split][m][n] = sum over the split's K blocks
  kEpiSwiGLU = 1,  // interleaved gate/up columns -> silu(g)*u -> Q8_0 codes + scales
  kEpiDots = 2,    // debug: also write every block's int32 dot to dots[m][n][b]
};

struct GemmPlan {
  int bn = 128;
  int splits = 1;
};

// Choose the N tile and the split-K factor for an M x N x nb problem.
GemmPlan gemm_plan(int64_t M, int64_t N, int nb, int num_sms, bool allow_split);

// y = A . B^T on the tensor cores.  A: activations (rows = M), B: weights
// (rows = N).  Epilogue kEpiF32 writes split s to out + s * split_stride.
// kEpiSwiGLU expects B rows interleaved in groups of kSwiGluGroup gate /
// kSwiGluGroup up rows and
// writes codes [M][ldq] fp16 and scales [nbF][ldqs] f32; with `out` set it
// also writes the f32 values it quantized to out [M][ldo] (debug capture).
struct GemmLaunch {
  GemmOperand A, B;
  int64_t M = 0, N = 0;
  int epi = kEpiF32;
  GemmPlan plan;
  float* out = nullptr;
  int64_t ldo = 0, split_stride = 0;
  __half* q_out = nullptr;
  int64_t ldq = 0;
  float* qs_out = nullptr;
  int64_t ldqs = 0;
  int64_t n_out_cols = 0;  // kEpiSwiGLU: padded count of SwiGLU outputs
  int32_t* dots = nullptr;
  int* err = nullptr;
  // B (codes and scales) is written by no kernel that may still be running
  // (weights uploaded before the call): the first stages' B loads then start
  // before the wait for the previous kernel of the stream
  bool b_static = false;
  // test hook (off by default): the time limit of every bounded wait (0: the
  // default) and one K stage that CTA 0's producer withholds (-1: none), so
  // that the MMA issuer's wait on it runs out
  uint64_t wait_ns = 0;
  int skip_stage = -1;
};

// Tensor maps are built once per (buffer, shape) and cached by the caller.
struct GemmMaps {
  CUtensorMap a, b, sa, sb;
};
int gemm_make_maps(const GemmOperand& A, const GemmOperand& B, int bn, GemmMaps* maps);
// A 2-D TMA map over a row-major [outer][inner] array of fp16 (or f32), box
// [box_outer][box_inner], 128-byte swizzle or none.  0 on success.
int tensor_map_2d(CUtensorMap* map, const void* base, bool f32, uint64_t inner, uint64_t outer,
                  uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128);
cudaError_t gemm_launch(const GemmLaunch& g, const GemmMaps& maps, int num_sms,
                        cudaStream_t stream);

// ---------------------------------------------------------------- row kernels
// RMSNorm (optional) then Q8_0 of rows; optionally first h += sum of split
// partials.  Writes fp16 codes [rows][ldq] + f32 scales [nb][ldqs] (GEMM
// layout) or int8 codes + f32 scales [rows][nb] (GEMV layout).
struct RowQuantArgs {
  float* h = nullptr;             // [rows][n] residual stream (read; written if nsplit > 0)
  const float* partials = nullptr;  // [nsplit][rows][n]
  int nsplit = 0;
  int64_t split_stride = 0;
  const float* norm_w = nullptr;  // nullptr: no RMSNorm
  float eps = 0.f;
  int64_t rows = 0, n = 0;
  int64_t row_offset = 0;  // first row of h / partials processed
  __half* q16 = nullptr;   // GEMM codes [rows][ldq]
  int64_t ldq = 0;
  float* s16 = nullptr;    // GEMM scales [nb][ldqs]
  int64_t ldqs = 0;
  int8_t* q8 = nullptr;    // GEMV codes [rows][nb*32]
  float* s8 = nullptr;     // GEMV scales [rows][nb]
  uint16_t* s8_bits = nullptr;  // optional fp16 bits [rows][nb] (tests)
};
cudaError_t row_quant_launch(const RowQuantArgs& a, cudaStream_t stream);

// h[t][:] = dequantized tok_embd row ids[t] (int8 codes + f32 scales).
cudaError_t embed_launch(const int8_t* emb_q, const float* emb_s, int64_t kpad, int nb,
                         const int32_t* ids, int nt, int64_t H, int n_vocab, float* h,
                         cudaStream_t stream);

// Device validation of ids/positions: writes MINFER error code into *status
// (0 when valid).  seen: n_ctx-bit scratch bitmap, cleared here first.
cudaError_t validate_launch(const int32_t* ids, const int32_t* pos, int nt, int n_vocab,
                            int n_ctx, uint32_t* seen, int* status, cudaStream_t stream);

// RoPE + KV store.  qkv = bias + sum of nsplit partials [nt][nq + 2 nkv] ...
struct RopeStoreArgs {
  const float* partials = nullptr;
  int nsplit = 1;
  int64_t split_stride = 0;
  const float* bias = nullptr;  // [(nh + 2 nkv) hd]
  const int32_t* pos = nullptr;
  int nt = 0, nh = 0, nkv = 0, hd = 0;
  int n_ctx = 0;                 // rows of the regions and of the cos/sin tables
  const float* cos_t = nullptr;  // [n_ctx][hd/2]
  const float* sin_t = nullptr;
  float* q_out = nullptr;  // [nt][nh*hd]; null: only the fp16 planes of Q are written
  float* kreg = nullptr;   // [n_ctx][nkv*hd]
  float* vreg = nullptr;
  __half* shadow[4] = {nullptr, nullptr, nullptr, nullptr};  // fp16 hi/lo copies of K, V
  __half* vt[2] = {nullptr, nullptr};  // fp16 hi/lo of V transposed: [nkv*hd][vt_ld] (key-major)
  int64_t vt_ld = 0;
  __half* q_planes[2] = {nullptr, nullptr};  // optional fp16 hi/lo of the rotated Q [nt][nh*hd]
  const int* status = nullptr;  // the model's two status words: no region write unless both are 0
  // Qwen3 QK-norm (null: none): per-head RMSNorm weights [hd] of Q and of K
  const float* q_norm = nullptr;
  const float* k_norm = nullptr;
  float eps = 0.f;
};
cudaError_t rope_store_launch(const RopeStoreArgs& a, cudaStream_t stream);
struct GemvArgs;
// One token, no QK-norm: the QKV GEMV (g: y = the raw Q|K|V sums) and the
// RoPE/store of r (partials = g.y, nsplit 1) in one kernel.
cudaError_t gemv_rope_launch(const GemvArgs& g, const RopeStoreArgs& r, cudaStream_t stream);

// Causal GQA attention of query rows [r0, r1) over the fp16 hi/lo shadow
// planes of a layer's K/V regions, split along the keys (ksplit keys per
// split, a multiple of 32), then merged, normalized and quantized.
struct AttnArgs {
  const float* q = nullptr;  // [nt][nh*hd]
  const int32_t* pos = nullptr;
  int r0 = 0, r1 = 0;
  const __half* shadow[4] = {nullptr, nullptr, nullptr, nullptr};  // K hi, K lo, V hi, V lo [n_ctx][nkv*hd]
  const __half* vt[2] = {nullptr, nullptr};  // V hi, V lo transposed [nkv*hd][vt_ld]
  int64_t vt_ld = 0;                         // >= n_ctx, a multiple of 64
  const __half* qp[2] = {nullptr, nullptr};  // Q hi, Q lo [r1][nh*hd] (tensor-core kernel)
  int nh = 0, nkv = 0, hd = 0;
  int n_ctx = 0;   // positions are clamped into [0, n_ctx) before any region read
  int nsplit = 1;  // key splits (CTAs per cluster), 1..8
  // One-row calls (r1 - r0 == 1) run the CUDA-core kernel of one thread-block
  // cluster per KV head when the f32 K/V regions [n_ctx][nkv*hd] are given
  // (16-byte aligned).
  const float* kreg = nullptr;
  const float* vreg = nullptr;
  // One-row kernel: the region rows below the query's position were written
  // by earlier calls (a single-token call), not by a kernel that may still be
  // running, so the first chunk of them loads before the grid wait.
  int kv_static_below = 0;
};
// Where the attention output goes: Q8_0 codes in the GEMM layout (q16 [rows][ldq]
// fp16 + s16 [nb][ldqs]) or the GEMV layout (q8 [rows][nb*32] + s8 [rows][nb]);
// output row index = query row - row_base.  f32 (optional): [nt][nh*hd].
struct AttnOut {
  __half* q16 = nullptr;
  int64_t ldq = 0;
  float* s16 = nullptr;
  int64_t ldqs = 0;
  int8_t* q8 = nullptr;
  float* s8 = nullptr;
  int64_t row_base = 0;
  float* f32 = nullptr;
};
// The tensor-core attention (k_attn_tc.cu) for calls of 64 rows and more with
// head_dim 64 or 128: one CTA per (128 rows, query head, key split); err is the
// device status word of timed-out waits.
bool attention_tc_supported(const AttnArgs& a);
// Whether the forward picks it: from one full 128-row tile on.
bool attention_tc_preferred(int rows, int nh, int num_sms);
cudaError_t attention_tc_launch(const AttnArgs& a, const AttnOut& out, int num_sms, int* err,
                                cudaStream_t stream);
// Key splits for `rows` query rows: enough CTAs to fill the GPU about twice.
int attention_nsplit(int rows, int nkv, int num_sms, int G);
cudaError_t attention_launch(const AttnArgs& a, const AttnOut& out, cudaStream_t stream);
// f32 K/V rows row0.. (count = rows * kvw values) -> fp16 hi/lo planes
// (planes[0..3] = K hi, K lo, V hi, V lo, pointing at row row0) and the
// transposed V planes vt[0..1] [kvw][vt_ld] at columns row0...
// x [count] f32 -> fp16 hi = rn(x), lo = rn(x - hi).
cudaError_t split_planes_launch(const float* x, int64_t count, __half* hi, __half* lo,
                                cudaStream_t stream);
cudaError_t kv_shadow_launch(const float* k, const float* v, int64_t count, __half* const* planes,
                             __half* const* vt, int64_t vt_ld, int row0, int kvw,
                             cudaStream_t stream);

// One-row quantized GEMV: y[n] = sum_b dw[n][b] * da[b] * dot_b (+ resid[n]).
// W int8 [N][kpad] + f32 scales [N][nb]; x int8 [kpad] + f32 scales [nb].
struct GemvArgs {
  const int8_t* wq = nullptr;
  const float* ws = nullptr;
  int64_t N = 0;
  int nb = 0;
  int64_t kpad = 0;
  const int8_t* xq = nullptr;
  const float* xs = nullptr;
  float* y = nullptr;
  const float* resid = nullptr;  // y = resid + W.x when set (may alias y)
  const int* status = nullptr;   // the model's two status words: no write of y unless both are 0
  int num_sms = 152;             // rows per warp are chosen to give every SM two CTAs
  // Fused one-row epilogues (q8 [nb*32] codes + s8 [nb] f32 scales of the result):
  // swiglu: rows are gate/up interleaved in groups of 32 (N = 2 * F padded to
  //   a multiple of 64); q8/s8 get the Q8_0 of silu(gate) * up; y is not written.
  // norm_w: y is written, then the last CTA to finish writes the Q8_0 of
  //   RMSNorm(y) * norm_w (eps) into q8/s8; ticket: a zero-initialized counter,
  //   left at zero.  Needs gemv_norm_fusable().
  int swiglu = 0;
  const float* norm_w = nullptr;
  float eps = 0.f;
  int8_t* q8 = nullptr;
  float* s8 = nullptr;
  unsigned* ticket = nullptr;
  // the weights are written by no kernel that may still be running (uploaded
  // before the call): the first round of weight loads then starts before the
  // wait for the previous kernel of the stream
  int w_static = 0;
};
cudaError_t gemv_launch(const GemvArgs& a, cudaStream_t stream);
// Whether a norm can ride the GEMV's last CTA: whole Q8_0 blocks, N <= 4096,
// 16-byte aligned y and norm_w, 4-byte aligned q8.
bool gemv_norm_fusable(int64_t N, const float* y, const float* norm_w, const int8_t* q8);

// int8 [rows][nb*32] + f32 [rows][nb] (GEMV layout) -> fp16 codes + block-major scales.
cudaError_t gemv_to_gemm_launch(const int8_t* q, const float* sc, int64_t rows, int nb,
                                __half* codes, float* scales, int64_t rows_pad, cudaStream_t stream);
// dst[0:n] = src[0:n] when both status words are 0.
cudaError_t copy_if_ok_launch(const float* src, float* dst, int64_t n, const int* status,
                              cudaStream_t stream);

// ---------------------------------------------------------------- load-time kernels
// f32 rows -> Q8_0 (int8 codes [rows][nb*32] + fp16 scale bits [rows][nb]).
cudaError_t quantize_rows_launch(const float* x, int64_t rows, int64_t n, int8_t* q,
                                 uint16_t* dbits, cudaStream_t stream);
// 34-byte Q8_0 blocks -> int8 codes + fp16 bits.
cudaError_t unpack_q8_0_launch(const uint8_t* blocks, int64_t rows, int64_t n, int8_t* q,
                               uint16_t* dbits, cudaStream_t stream);
// int8 codes + fp16 bits (rows [src_row0, +rows)) -> GEMM planes: fp16 codes
// at dst rows given by row_map (row r -> dst_row(r)) and f32 scales [nb][dst_rows_pad].
struct RepackArgs {
  const int8_t* q = nullptr;
  const uint16_t* dbits = nullptr;
  int64_t rows = 0;
  int nb = 0;
  __half* dst_codes = nullptr;  // [dst_rows][nb*32]
  float* dst_scales = nullptr;  // [nb][dst_rows_pad]
  int64_t dst_rows_pad = 0;
  int64_t dst_row0 = 0;     // destination row of source row 0 (plain layout)
  int interleave = 0;       // 1: gate (which=0) / up (which=1) interleave in groups of kSwiGluGroup
  int which = 0;
};
cudaError_t repack_gemm_launch(const RepackArgs& a, cudaStream_t stream);
// int8 codes + fp16 bits -> GEMV planes (int8 codes copy + f32 scales [rows][nb]);
// interleave = 1: source row r lands on row (r / 32) * 64 + which * 32 + r % 32
// (the fused SwiGLU GEMV's gate/up layout).
cudaError_t repack_gemv_launch(const int8_t* q, const uint16_t* dbits, int64_t rows, int nb,
                               int8_t* dst_q, float* dst_s, int interleave, int which,
                               cudaStream_t stream);
// GEMM planes -> canonical int8 codes / fp16 bits (tests).
cudaError_t gemm_plane_to_q8_launch(const __half* codes, const float* scales, int64_t rows,
                                    int64_t rows_pad, int nb, int8_t* q, uint16_t* dbits,
                                    cudaStream_t stream);

// Split-partials sum: out[m][n] = sum_s partials[s][m][n].
cudaError_t sum_splits_launch(const float* partials, int nsplit, int64_t split_stride,
                              int64_t count, float* out, cudaStream_t stream);

}  // namespace minfer
