/*
 * minfer.h -- C ABI of the GB300 (sm_103a) prefill library.
 *
 * One call, minfer_prefill, runs the prefill forward of a Qwen2-style decoder
 * over a whole prompt: every token goes through every layer in one pass, K/V
 * rows land in persistent per-layer regions at the rows named by a positions
 * buffer, attention is causal (token t sees positions 0..=pos[t]), and only
 * the last token's logits come back ("09 · Prefill: the first forward",
 * sections 2.2-2.4; "05 · Graph build — the IR and the builder", section 2.5
 * node list and section 2.8 tail rows).  Weights are Q8_0 (32 int8 codes and
 * one fp16 scale per block) and every matmul input activation is quantized
 * to Q8_0 on the fly (walkthrough index, master table, row "CPU matmul
 * kernels").
 *
 * Conventions
 *  - Every function returns MINFER_OK (0) or a negative MINFER_ERR_* code;
 *    minfer_strerror() names it.
 *  - "host" pointers are ordinary CPU memory, "device" pointers are CUDA
 *    global memory on the current device.  Pointers are borrowed for the
 *    duration of the call only, unless stated otherwise.
 *  - Matrices use the GGUF convention of the pages ("05 · Graph build",
 *    section 2.4): ne0 is the contiguous (input) dimension, ne1 the number of
 *    rows (output dimension); memory is row-major [ne1][ne0].
 *  - Arguments are validated on the host before any device write; a call
 *    that fails validation leaves the KV regions and the logits untouched.
 *  - A model and the KV handles made from it belong to the CUDA device that
 *    was current at minfer_model_create; call them with that device current.
 *    One call at a time per (model, kv) pair.
 */
#ifndef MINFER_H
#define MINFER_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- errors */
#define MINFER_OK 0
#define MINFER_ERR_ARG (-1)            /* null pointer, bad size, duplicate position */
#define MINFER_ERR_POS_OOB (-2)        /* a position < 0 or >= the KV region's n_ctx */
#define MINFER_ERR_TOKEN_OOB (-3)      /* a token id < 0 or >= n_vocab */
#define MINFER_ERR_MISSING_TENSOR (-4) /* a tensor the forward needs was never set */
#define MINFER_ERR_SHAPE (-5)          /* unknown tensor name, wrong ne0/ne1/type, or hparams
                                          the kernels are not built for */
#define MINFER_ERR_CUDA (-6)           /* a CUDA runtime/driver call failed */
#define MINFER_ERR_OOM (-7)            /* device allocation failed */
#define MINFER_ERR_DEVICE (-8)         /* a kernel gave up a bounded wait (status word set) */
#define MINFER_ERR_STATE (-9)          /* call order violated (e.g. prefill before finalize) */
#define MINFER_ERR_TOO_LARGE (-10)     /* the problem does not fit a fixed-size scratch area */

/* Device status codes (minfer_device_status): which bounded wait of which
 * kernel gave up first when a call returned MINFER_ERR_DEVICE. */
#define MINFER_DEV_OK 0
#define MINFER_DEV_TIMEOUT_TMA_EMPTY 1 /* GEMM producer waiting for a free operand stage */
#define MINFER_DEV_TIMEOUT_MMA_FULL 2  /* GEMM MMA issuer waiting for a loaded operand stage */
#define MINFER_DEV_TIMEOUT_MMA_SLOT 3  /* GEMM MMA issuer waiting for a free TMEM slot */
#define MINFER_DEV_TIMEOUT_EPILOGUE 4  /* GEMM epilogue waiting for scales or a finished slot */
#define MINFER_DEV_TIMEOUT_DRAIN 5     /* GEMM draining its copies and MMAs after a timeout */
#define MINFER_DEV_TIMEOUT_ATTN 6      /* tensor-core attention, any of its waits */

/* ---------------------------------------------------------------- tensors */
#define MINFER_F32 0  /* float32 values */
#define MINFER_Q8_0 8 /* blocks of 34 bytes: uint16 fp16 scale bits (little endian),
                         then 32 int8 codes; a row of ne0 values holds ceil(ne0/32)
                         blocks, the missing tail elements of a partial block are 0 */

typedef struct minfer_hparams {
  int n_layer;       /* transformer layers */
  int n_embd;        /* hidden width H */
  int n_head;        /* query heads */
  int n_head_kv;     /* key/value heads; n_head % n_head_kv == 0 */
  int head_dim;      /* dims per head: 64 or 128 (the two widths the attention
                        kernels are built for; minfer_model_create rejects others
                        with MINFER_ERR_SHAPE) */
  int n_ff;          /* FFN width F */
  int n_vocab;       /* vocabulary V */
  int max_seq_len;   /* upper clamp of n_ctx ("09 · Prefill", section 2.5) */
  float rope_theta;  /* RoPE frequency base */
  float rms_eps;     /* RMSNorm epsilon */
  int tied_embeddings; /* 1: lm_head reuses token_embd.weight */
  int qk_norm;       /* 1: Qwen3 -- each head of Q and K is RMS-normalized over head_dim
                        (weights blk.{i}.attn_q_norm.weight / attn_k_norm.weight,
                        head_dim entries each) after the bias and before RoPE
                        ("05 · Graph build", section 2.5: qk_norm; section 3.2:
                        FusedQkvNorm); the Q/K/V biases are then optional (zero
                        when absent).  0: Qwen2, biases required. */
} minfer_hparams;

typedef struct minfer_tensor {
  const char* name; /* GGUF names: token_embd.weight, output_norm.weight, output.weight,
                       blk.{i}.{attn_norm.weight, attn_q.weight, attn_q.bias,
                       attn_k.weight, attn_k.bias, attn_v.weight, attn_v.bias,
                       attn_output.weight, ffn_norm.weight, ffn_gate.weight,
                       ffn_up.weight, ffn_down.weight}; with qk_norm also
                       blk.{i}.{attn_q_norm.weight, attn_k_norm.weight} */
  int type;         /* MINFER_F32 (vectors and matrices) or MINFER_Q8_0 (matrices) */
  int64_t ne0, ne1; /* ne0 contiguous; ne1 = 1 for vectors */
  const void* data; /* host memory, borrowed during the call */
} minfer_tensor;

typedef struct minfer_model minfer_model;
typedef struct minfer_kv minfer_kv;

/* ---------------------------------------------------------------- model */

/* Create an empty model on the current device ("09 · Prefill", section 3.1:
 * the model is its hparams plus weight tensors registered by name).  *out is
 * owned by the caller and released with minfer_free.  MINFER_ERR_ARG for a
 * non-positive size or n_head not a multiple of n_head_kv; MINFER_ERR_SHAPE
 * for shapes the kernels are not built for: head_dim other than 64 or 128,
 * more than 8 query heads per KV head, n_embd or n_head*head_dim above 4096;
 * MINFER_ERR_CUDA without a CUDA device. */
int minfer_model_create(const minfer_hparams* hp, minfer_model** out);

/* Register one weight tensor under its GGUF name ("05 · Graph build",
 * section 3.1: the builder refers to weights by name only, e.g.
 * "blk.7.attn_q.weight", and the backend resolves the name to a registered
 * buffer).  The tensor is copied to the device: F32 matrices are quantized to
 * Q8_0 on the device (same block rule as the activations); Q8_0 matrices are
 * taken as given; matrices are repacked into the tensor-core layout.  Host
 * data may be freed on return.  MINFER_ERR_SHAPE for an unknown name or a
 * shape or type that does not match hp. */
int minfer_model_set_tensor(minfer_model* m, const minfer_tensor* t);

/* Check that every tensor is present (MINFER_ERR_MISSING_TENSOR otherwise,
 * the pages' "missing weight name is an execution-time error", "05 · Graph
 * build", section 3.4 item 8) and make the model ready for prefill. */
int minfer_model_finalize(minfer_model* m);

/* create + set every tensor + finalize in one call: the weights registered
 * by GGUF name ("09 · Prefill", section 3.1; "05 · Graph build", section 3.1)
 * and checked complete ("05 · Graph build", section 3.4 item 8: a weight
 * name with no registered tensor is an error).  On failure *out is NULL and
 * nothing stays allocated. */
int minfer_load_weights(const minfer_hparams* hp, const minfer_tensor* tensors, int n,
                        minfer_model** out);

/* Release a model and every device buffer it holds (weights, workspace,
 * recorded graphs).  The weights live for the whole run of the pages' engine
 * ("09 · Prefill", section 3.1: the model with its registered tensors is an
 * input of every forward); this ends that lifetime.  KV handles made from the
 * model must be freed first.  NULL is ignored. */
void minfer_free(minfer_model* m);

/* ---------------------------------------------------------------- KV regions */

/* Per-layer K and V regions of n_ctx rows x (n_head_kv * head_dim) f32,
 * zero-filled, sized once ("09 · Prefill", section 2.5: n_ctx clamped to
 * max_seq_len, regions never resized).  *out owned by the caller. */
int minfer_kv_create(minfer_model* m, int n_ctx, minfer_kv** out);
/* The n_ctx the regions were sized with ("09 · Prefill", section 2.5). */
int minfer_kv_n_ctx(const minfer_kv* kv);
/* Release the regions.  They persist across prefill calls by design ("09 ·
 * Prefill", section 3.1: the filled KV cache is the call's second output and
 * every later call reads it; section 2.5: regions survive graph rebuilds);
 * this ends their lifetime.  NULL is ignored. */
void minfer_kv_free(minfer_kv* kv);

/* Copy rows [row0, row0 + nrows) of layer `layer`'s K (which = 0) or V
 * (which = 1) region to/from host memory (nrows x n_head_kv*head_dim f32).
 * Synchronous.  For tests, snapshots and canaries: the per-layer KV dumps
 * that start a CPU-vs-GPU comparison ("09 · Prefill", section 4,
 * MINFER_GRAPH_DUMP) and the row layout of section 2.2 (row p holds position
 * p).  MINFER_ERR_ARG for a layer, which or row range outside the regions. */
int minfer_kv_read(const minfer_kv* kv, int layer, int which, int row0, int nrows, float* out);
int minfer_kv_write(minfer_kv* kv, int layer, int which, int row0, int nrows, const float* in);

/* ---------------------------------------------------------------- prefill */

/* The prefill forward ("09 · Prefill", section 3.2, forward_cached: preflight,
 * fill inputs, execute, one copy of the logits out).
 *   token_ids[n_tokens], positions[n_tokens]: host int32; positions distinct
 *     and within [0, n_ctx) of kv.
 *   logits_out: host, n_vocab floats, caller-owned; written exactly once on
 *     success with the last token's logits, never on failure.
 * K/V rows positions[t] of every layer are overwritten; every other row is
 * left untouched.  Synchronous: returns when the logits are in logits_out. */
int minfer_prefill(minfer_model* m, const int32_t* token_ids, const int32_t* positions,
                   int n_tokens, minfer_kv* kv, float* logits_out);

/* Same forward with device-resident inputs and output, enqueued on `stream`
 * (a cudaStream_t, or NULL for the model's own stream) without a host sync
 * ("09 · Prefill", section 3.2: fill the input buffers, execute; "05 · Graph
 * build", section 2.7: one recorded launch sequence per shape, replayed).
 * d_token_ids, d_positions: device int32[n_tokens]; d_logits: device
 * float[n_vocab].  Positions and ids are validated on the device: when one is
 * out of range or a position repeats, no K/V row and no logit is written and
 * the error is reported by the next minfer_sync_status.  The launch sequence
 * is recorded once per (n_tokens, kv) as a CUDA graph and replayed. */
int minfer_prefill_device(minfer_model* m, const int32_t* d_token_ids,
                          const int32_t* d_positions, int n_tokens, minfer_kv* kv,
                          float* d_logits, void* stream);

/* Several logits rows ("09 · Prefill", section 2.4: n_out; "05 · Graph
 * build", section 2.8: the last layer keeps the tail n_out rows): the logits
 * of the last n_out tokens, in token order, into logits_out [n_out][n_vocab]
 * (host) or d_logits (device).  1 <= n_out <= n_tokens, else MINFER_ERR_ARG.
 * n_out = 1 is minfer_prefill / minfer_prefill_device.  With n_out > 1 the
 * last layer carries its tail rows on the tensor cores and the lm_head runs
 * as one GEMM; its tensor-core copy of the lm_head weights is built on the
 * first such call. */
int minfer_prefill_n(minfer_model* m, const int32_t* token_ids, const int32_t* positions,
                     int n_tokens, minfer_kv* kv, int n_out, float* logits_out);
int minfer_prefill_device_n(minfer_model* m, const int32_t* d_token_ids,
                            const int32_t* d_positions, int n_tokens, minfer_kv* kv, int n_out,
                            float* d_logits, void* stream);

/* Wait for the work enqueued by minfer_prefill_device on `stream` and return
 * its status (MINFER_OK, MINFER_ERR_POS_OOB, MINFER_ERR_TOKEN_OOB,
 * MINFER_ERR_ARG or MINFER_ERR_DEVICE): the preflight check of "09 ·
 * Prefill", section 3.4, reported after the fact for device-resident
 * inputs. */
int minfer_sync_status(minfer_model* m, void* stream);

/* ---------------------------------------------------------------- debug hooks */

/* Register a host buffer that the next prefill calls fill with hidden states:
 * (n_layer + 1) slots of [n_tokens][n_embd] f32, slot 0 the embedding, slot
 * l + 1 the output of layer l; the last layer carries only the last token
 * (written to row 0 of its slot).  NULL disables.  The buffer is borrowed
 * until disabled ("09 · Prefill", section 4: per-layer dumps for
 * CPU-vs-GPU comparison). */
int minfer_set_dump(minfer_model* m, float* host_hidden, int max_tokens);

/* Copy a named activation buffer of the last prefill to host memory
 * (synchronous, debugging; "09 · Prefill", section 4: per-node dumps for
 * offline comparison): "h" f32 [nt][n_embd], "att" f32 [nt][n_head*hd]
 * (attention output; the last layer writes only its last row), "xf" fp16
 * codes [nt][ceil(n_ff/32)*32] (quantized SwiGLU output of the layer before
 * last), "xf_s" f32 scales [ceil(n_ff/32)][ceil(nt/128)*128].  bytes is the
 * host buffer size; MINFER_ERR_ARG for an unknown name or a short buffer. */
int minfer_debug_read(minfer_model* m, const char* buffer, void* host, int64_t bytes);

/* Capture the intermediates of layer `layer` (0 <= layer < n_layer; -1 turns
 * it off) during the next prefill calls, which then run without the graph
 * ("09 · Prefill", section 4: per-node and per-layer dumps of the live
 * forward; "05 · Graph build", section 2.5: the node list they follow).
 * minfer_debug_read then also serves, for the last captured call (nt rows,
 * ntp = ceil(nt/128)*128, kx = ceil(n_embd/32)*32), the buffers below; the
 * last layer, which carries only the final token past its K/V projections,
 * captures h_in, x_codes, x_scales and qkv alone:
 *   "h_in", "h_mid", "h_out"  f32 [nt][n_embd]: residual stream entering the
 *                             layer, after the attention residual, leaving it
 *   "x_codes", "f_codes"      fp16 [nt][kx]: Q8_0 codes of attn_norm(h_in) and
 *                             ffn_norm(h_mid); "x_scales", "f_scales" f32
 *                             [kx/32][ntp] (block-major)
 *   "qkv"                     f32 [nt][(n_head + 2 n_head_kv) head_dim]: Q|K|V
 *                             projections before bias and RoPE
 *   "qrot"                    f32 [nt][n_head*head_dim]: rotated Q
 *   "att_codes", "att_scales" Q8_0 of the attention output (fp16 [nt][q],
 *                             f32 [q/32][ntp]); "att" its f32 values [nt][q]
 *   "s_codes", "s_scales"     Q8_0 of the SwiGLU output (fp16 [nt][ceil(n_ff/32)*32],
 *                             f32 [ceil(n_ff/32)][ntp])
 *   "s_f32"                   f32 [nt][ceil(n_ff/32)*32]: the values silu(g)*u
 *                             that the gate/up GEMM's epilogue quantized into
 *                             "s_codes" (written by that same epilogue)
 * A single-token call (one-row GEMV path) captures instead, one row each:
 * "h_in", "h_mid", "h_out", "qkv", "qrot", "att" (f32) and the Q8_0 inputs
 * of its GEMVs as int8 codes + f32 scales: "x_q8"/"x_s8" (attn_norm),
 * "att_q8"/"att_s8", "f_q8"/"f_s8" (ffn_norm), "s_q8"/"s_s8" (SwiGLU).
 * Returns MINFER_ERR_ARG for a layer out of range; a failed capture
 * allocation fails the prefill call with MINFER_ERR_CUDA. */
int minfer_debug_layer(minfer_model* m, int layer);

/* Per-kernel device time of the prefill calls since the last reset ("09 ·
 * Prefill", section 4: the bench's per-stage timing), measured
 * with CUDA events around each launch: kernel class k in [0, n) gets its
 * name, its launch count and its total milliseconds.  enable = 1 turns the
 * events on (they add a few microseconds per launch), 0 off. */
int minfer_profile_enable(minfer_model* m, int enable);
int minfer_profile_read(minfer_model* m, int k, const char** name, int64_t* launches,
                        double* total_ms);

/* ---------------------------------------------------------------- single stages
 * Each stage of the forward on its own, device pointers, synchronous, for
 * parity tests.  Codes are int8 [rows][nb*32] (nb = ceil(n/32)), scale bits
 * uint16 fp16 [rows][nb].  They run the same kernels as minfer_prefill. */

/* Q8_0-quantize rows of x [rows][n] (walkthrough index, "CPU matmul kernels"). */
int minfer_op_quantize(const float* d_x, int64_t rows, int64_t n, int8_t* d_q, uint16_t* d_d);

/* RMSNorm then Q8_0 ("05 · Graph build", section 2.5: rms_norm, eps). */
int minfer_op_rmsnorm_quantize(const float* d_x, const float* d_w, int64_t rows, int64_t n,
                               float eps, int8_t* d_q, uint16_t* d_d);

/* y[M][N] = Q8_0(x) . Q8_0(W)^T on the tensor-core GEMM (walkthrough index,
 * master table, row "CPU matmul kernels": quantized weight times on-the-fly
 * Q8_0 activation); optional per-block int32 dots out [M][N][nb] (d_dots may
 * be NULL). x codes [M][nb*32], W codes [N][nb*32]; K = n columns. */
int minfer_op_gemm(const int8_t* d_xq, const uint16_t* d_xd, int64_t M, const int8_t* d_wq,
                   const uint16_t* d_wd, int64_t N, int64_t K, float* d_y, int32_t* d_dots);

/* Fused gate/up GEMM + SwiGLU + Q8_0: s = silu(x.Wg^T) * (x.Wu^T), then
 * quantized; Wg, Wu [F][nb*32]; outputs codes [M][ceil(F/32)*32] and scale
 * bits [M][ceil(F/32)]. ("05 · Graph build", section 2.5: SwiGLU). */
int minfer_op_gemm_swiglu(const int8_t* d_xq, const uint16_t* d_xd, int64_t M,
                          const int8_t* d_gq, const uint16_t* d_gd, const int8_t* d_uq,
                          const uint16_t* d_ud, int64_t F, int64_t K, int8_t* d_sq,
                          uint16_t* d_sd);

/* Causal GQA attention of query rows q [nt][n_head*head_dim] (already
 * rotated) over K/V regions [n_ctx][n_head_kv*head_dim]; token t sees region
 * rows 0..=pos[t] with scale 1/sqrt(head_dim) ("09 · Prefill", section 2.2;
 * "05 · Graph build", section 2.5). o [nt][n_head*head_dim] f32.  Calls of
 * 64 rows and more run the tensor-core kernel, shorter ones the mma.sync
 * kernel (the prefill uses the tensor-core kernel from 128 rows on), so the
 * stage tests reach both. */
int minfer_op_attention(const float* d_q, const int32_t* d_pos, int nt, const float* d_k,
                        const float* d_v, int n_ctx, int n_head, int n_head_kv, int head_dim,
                        float* d_o);

/* RoPE (NeoX half-split pairs, theta^(-2i/hd)) of the Q and K parts of
 * qkv [nt][(nh + 2 nkv) hd] plus bias, and the KV store: K/V regions row
 * pos[t] <- rotated K[t], V[t] ("09 · Prefill", section 2.2). q_out
 * [nt][nh*hd] f32. Positions must be valid for n_ctx. */
int minfer_op_rope_store(const float* d_qkv, const float* d_bias, const int32_t* d_pos, int nt,
                         int n_head, int n_head_kv, int head_dim, float theta, int n_ctx,
                         float* d_q_out, float* d_k, float* d_v);

/* The same with Qwen3 QK-norm between the bias and RoPE: each head of Q and
 * K is RMS-normalized over its head_dim values (mean of squares, eps added,
 * scale rounded to f32, then (x * scale) * w) with the weights d_qnorm /
 * d_knorm [head_dim] ("05 · Graph build", section 3.2: FusedQkvNorm).
 * d_bias may be NULL. */
int minfer_op_qknorm_rope_store(const float* d_qkv, const float* d_bias, const float* d_qnorm,
                                const float* d_knorm, float eps, const int32_t* d_pos, int nt,
                                int n_head, int n_head_kv, int head_dim, float theta, int n_ctx,
                                float* d_q_out, float* d_k, float* d_v);

/* Same product as minfer_op_gemm (same kernels, same split plan) without any
 * device allocation, for callers that cannot call cudaMalloc: a process whose
 * own memory pool reserved nearly all of HBM at start-up (a cudaMalloc would
 * fail, or take memory the pool counts on), and code that must not stall the
 * whole device (cudaFree, which an allocating call needs sooner or later,
 * synchronizes every stream of the device).
 *  - Scratch: the operand planes and the split-K partials live in one 32 MiB
 *    __device__ array inside the library, which every GPU that loads the
 *    library holds until the process exits.  A problem whose scratch does not
 *    fit (or with M, N or K above 2^31 - 1) returns MINFER_ERR_TOO_LARGE
 *    before any device work.
 *  - Set-up: the first call on each device looks up the array's device
 *    address and creates the library's own non-blocking stream for that
 *    device; make that first call before any stream capture.  Both are kept
 *    for the life of the process: do not use this entry point across a
 *    cudaDeviceReset of that device.
 *  - Ordering: the work runs on that non-blocking stream, and the call waits
 *    for that stream alone (no device-wide synchronization).  The caller's
 *    operands must be ready when the call starts (synchronize the stream that
 *    produced them first); d_y holds the result when the call returns.
 *  - Sharing: all calls share the array and find the previous call's contents
 *    there (what must start at zero is cleared on every call).  Calls whose
 *    work overlaps on the GPU race on it: do not call it from two threads at
 *    once.
 * The pages have no counterpart of this entry point. */
int minfer_op_gemm_noalloc(const int8_t* d_xq, const uint16_t* d_xd, int64_t M,
                           const int8_t* d_wq, const uint16_t* d_wd, int64_t N, int64_t K,
                           float* d_y);

/* ---------------------------------------------------------------- misc */
/* A static, NUL-terminated name of an error code (never NULL; "unknown error"
 * for codes outside the list).  The codes restate the pages' failures as
 * return values instead of aborts: a position at or past n_ctx ("09 ·
 * Prefill", section 3.4: the preflight assert and the store kernel's hard
 * error), a weight name never registered ("05 · Graph build", section 3.4
 * item 8). */
const char* minfer_strerror(int code);
/* Device-side status of the last failed call (a MINFER_DEV_* code, 0 if
 * none): which bounded wait of which kernel gave up when a call returned
 * MINFER_ERR_DEVICE ("09 · Prefill", section 3.4: a failure is reported
 * loudly, never as silently wrong output).  Once a wait has given up, the
 * later kernels of that call write no K/V row and no logit; rows written
 * before the failure point stay written. */
int minfer_device_status(minfer_model* m);

/* Test hook for that failure path, off by default ("09 · Prefill", section
 * 3.4: the failure must surface as an error, not as wrong output).  While
 * `layer` >= 0, the prefill calls of m run without the recorded graph, every
 * bounded wait of the GEMMs gives up after wait_limit_ns (> 0) instead of
 * 2 s, and the gate/up GEMM of that layer withholds one operand stage, so
 * that a wait on it runs out: the call returns MINFER_ERR_DEVICE and
 * minfer_device_status names the wait.  The K/V rows of that layer were
 * written before the failure point; later layers and the logits are not.  layer = -1 turns it off (the next
 * call runs normally).  MINFER_ERR_ARG for a layer out of range or a
 * non-positive limit. */
int minfer_debug_fault(minfer_model* m, int layer, int64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif
#endif /* MINFER_H */
