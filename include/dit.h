/*
 * dit.h -- C ABI of the GB300 diffusion-transformer hot path (libdit.so).
 *
 * The library computes the forward pass of one diffusion-transformer block
 * and the flow-matching Euler denoise step that repeats it, on one NVIDIA
 * GB300 (sm_103a), with hand-written CUDA kernels.
 *
 * Sources, cited by page title and section:
 *   [ERNIE]  "Porting ERNIE-Image-Turbo to Zig and Metal: An 8B Diffusion
 *            Transformer From Scratch on Apple Silicon"
 *   [ZFLOW]  "From Python + CUDA to Pure Rust + Metal 4: How zml-flow-rs Stops
 *            Us Writing a Kernel Per Model"
 *   [MAKEPAD] makepad commit log, libs/ai/metal/shaders/ggml (resident
 *            pre-norm ViT backbone)
 *
 * Conventions shared by every entry point:
 *   - Ownership: the caller allocates and owns every buffer.  No entry point
 *     allocates or frees memory, and none synchronises with the host except
 *     dit_last_device_error().
 *   - Pointers marked "device" must point to GPU memory of the current
 *     device; "host" pointers to CPU memory.  Device pointers must be 16-byte
 *     aligned and every row stride a multiple of 16 bytes (the tensor-memory
 *     copy engine requires it); violations return DIT_EINVAL.
 *   - Matrices are row-major.  Weights are bf16 and stored [out, in], so a
 *     linear computes y = x W^T.  In the W8A8 format (linear_format 1) the
 *     four projection weights are instead e4m3 codes of the rotated weights
 *     with one fp32 scale per row, made by dit_rotate_quantize.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  All
 *     work is enqueued asynchronously on it.
 *   - Empty inputs: the row-wise entry points (norms, coding, Euler) accept
 *     zero rows or elements, with any pointers (NULL included), check their
 *     scalar arguments and return DIT_OK without enqueuing anything; a block,
 *     a denoise step, an attention call or a linear with zero tokens or rows
 *     returns DIT_EINVAL.
 *   - Errors: invalid arguments return DIT_EINVAL and enqueue nothing; shapes
 *     outside the kernel set return DIT_EUNSUPPORTED; a failed launch returns
 *     DIT_ECUDA.  Kernels never trap: every wait inside a kernel is bounded,
 *     and a wait that runs out sets a device error word that
 *     dit_last_device_error() reports as DIT_ETIMEOUT.
 */
#ifndef DIT_H_
#define DIT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DIT_OK = 0,
  DIT_EINVAL = -1,
  DIT_EUNSUPPORTED = -2,
  DIT_EWORKSPACE = -3,
  DIT_ECUDA = -4,
  DIT_ETIMEOUT = -5
} dit_status;

/* Shape and semantics of one block ([ERNIE] section I: hidden 4096, 32 heads
 * x 128, 3D RoPE; [ZFLOW] section VI: the Backend op vocabulary with heads,
 * kv_heads, norm kind and rope layout as parameters). */
typedef struct {
  int32_t hidden;       /* H, multiple of 64 */
  int32_t n_heads;      /* query heads */
  int32_t n_kv_heads;   /* key/value heads; n_heads % n_kv_heads == 0 (GQA) */
  int32_t head_dim;     /* d: 64 or 128 */
  int32_t ffn;          /* F, SwiGLU width, multiple of 128 */
  int32_t rope_layout;  /* 0: pairs (2k, 2k+1) (DiT); 1: pairs (k, k+d/2) (ViT) */
  int32_t adaln;        /* 1: AdaLN modulation + gated residuals from mod[6,H];
                           0: pre-norm LayerNorm with gain/bias, plain residuals */
  int32_t qk_norm;      /* 1: per-head norm with gain/bias on q and k */
  float ln_eps;         /* norm epsilon (1e-6) */
  /* Variants ([ERNIE] section IV per-layer graph and section V, Bug 1;
   * [ZFLOW] sections IV and V); zero selects the default in brackets. */
  int32_t norm_kind;    /* [0] LayerNorm; 1 RMSNorm: pre-norms, qk-norm, final norm */
  int32_t glu_act;      /* [0] SiLU(gate) up; 1 GELU(gate) up, tanh form with the
                           argument clamped to +-20 and the output to +-65504 */
  int32_t rope_order;   /* [0] qk-norm then RoPE; 1 RoPE then qk-norm */
  int32_t gate_fn;      /* [0] x + g y; 1 x + tanh(g) y; 2 x + sigmoid(g) y */
  /* Format of the four projections ([ZFLOW] section VII, "W8A8Rot"):
   * [0] bf16 operands; 1 W8A8 with the H256 rotation: the activation rows
   * are rotated along K by the 256-point Hadamard matrix and coded in e4m3
   * with one scale per row inside the block, the weights arrive already
   * rotated and coded (dit_rotate_quantize).  Needs hidden, n_heads d and
   * ffn to be multiples of 256. */
  int32_t linear_format;
} dit_block_config;

enum { DIT_LINEAR_BF16 = 0, DIT_LINEAR_W8A8_H256 = 1 };

/* One block's weights, all device pointers.  Linears bf16 [out, in]:
 *   w_qkv  [(n_heads + 2 n_kv_heads) d, H]  rows: q heads, k heads, v heads
 *   w_o    [H, n_heads d]
 *   w_gu   [2F, H]   gate rows first, then up rows
 *   w_down [H, F]
 * Norm parameters fp32, 16-byte aligned: q_g, q_b, k_g, k_b [d] (used when
 * qk_norm); ln1_g, ln1_b, ln2_g, ln2_b [H] (used when adaln == 0).
 * With linear_format DIT_LINEAR_W8A8_H256 the four linears hold e4m3 codes
 * (one byte per element, same shapes) of the rotated weights and the four
 * scale pointers their fp32 per-row scales [rows]; otherwise the scales are
 * ignored. */
typedef struct {
  const void *w_qkv, *w_o, *w_gu, *w_down;
  const float *q_g, *q_b, *k_g, *k_b;
  const float *ln1_g, *ln1_b, *ln2_g, *ln2_b;
  const float *w_qkv_scale, *w_o_scale, *w_gu_scale, *w_down_scale;
} dit_block_weights;

/* The denoiser around the blocks ([ERNIE] section IV: latent [4096,128] ->
 * patch embed -> 36 blocks -> final AdaLN norm -> projection back to the
 * latent channels). */
typedef struct {
  dit_block_config block;
  int32_t n_layers;
  int32_t latent_channels;  /* C (128) */
  int32_t t_dim;            /* sinusoid width (256); a multiple of 8, <= 16384 */
  float t_scale;            /* timestep T = t_scale * sigma (1000) */
  int32_t rope_axes[3];     /* per-axis RoPE widths, sum = head_dim ([32,48,48]) */
  float rope_theta;         /* 256 */
} dit_model_config;

/* Head/tail weights (device) and the per-layer block weights (a HOST array of
 * n_layers structs, each holding device pointers).
 *   patch_w bf16 [H, C], patch_b fp32 [H]
 *   t_w1 bf16 [H, t_dim], t_b1 [H];  t_w2 bf16 [H, H], t_b2 [H]
 *   mod_w bf16 [6H, H], mod_b [6H]    -> [shift1,scale1,gate1,shift2,scale2,gate2]
 *   fin_w bf16 [2H, H], fin_b [2H]    -> [scale, shift] of the final norm
 *   out_w bf16 [C, H], out_b [C] */
typedef struct {
  const void* patch_w; const float* patch_b;
  const void* t_w1; const float* t_b1;
  const void* t_w2; const float* t_b2;
  const void* mod_w; const float* mod_b;
  const void* fin_w; const float* fin_b;
  const void* out_w; const float* out_b;
  const dit_block_weights* layers;
} dit_model_weights;

/* ------------------------------------------------------------------ the path */

/* Bytes of device workspace dit_block_forward needs for n_tokens tokens in
 * n_seqs independent sequences.  0 on invalid arguments. */
size_t dit_block_workspace_bytes(const dit_block_config* cfg, int32_t n_tokens,
                                 int32_t n_seqs);

/* One transformer block, in place on the fp32 residual stream
 * ([ERNIE] section IV, per-layer graph; [MAKEPAD] pre-norm ViT block):
 *   a = LN(x) (1 + scale1) + shift1            (adaln; else LN(x) g1 + b1)
 *   q, k, v = a Wqkv^T;  q, k <- LN_d(.) g + b  (qk_norm), then RoPE
 *   o = softmax(q k^T / sqrt(d)) v              non-causal, per sequence, GQA
 *   x <- x + gate1 (o Wo^T)                     (gate 1 when adaln == 0)
 *   a = LN(x) (1 + scale2) + shift2
 *   x <- x + gate2 (SiLU(a Wg^T) (a Wu^T)) Wd^T
 * x:   device fp32 [n_tokens, H], read and overwritten.
 * n_seqs: tokens are n_seqs sequences of n_tokens / n_seqs rows; attention
 *      stays inside a sequence.
 * mod: device fp32 [6, H] (adaln) or NULL.
 * rope_cos, rope_sin: device fp32 [head_dim / 2, n_tokens / n_seqs]
 *      (pair-major), entry (k, t) the rotation of pair k of the token at
 *      position t of its sequence (see dit_rope_table_grid /
 *      dit_rope_table_vit).
 * workspace: device, >= dit_block_workspace_bytes(), else DIT_EWORKSPACE. */
dit_status dit_block_forward(const dit_block_config* cfg, const dit_block_weights* w,
                             float* x, int32_t n_tokens, int32_t n_seqs,
                             const float* mod, const float* rope_cos,
                             const float* rope_sin, void* workspace, size_t ws_bytes,
                             void* stream);

/* Bytes of device workspace dit_denoise_step needs. */
size_t dit_denoise_workspace_bytes(const dit_model_config* cfg, int32_t grid_h,
                                   int32_t grid_w, int32_t n_txt);

/* One flow-matching Euler step of the whole denoiser ([ERNIE] section IV and
 * the 8-step loop around it; [ZFLOW] section IV, Euler sign +1):
 *   e = [cos(T w), sin(T w)], T = t_scale sigma;  temb = W2 SiLU(W1 e + b1) + b2
 *   mod = Wm SiLU(temb) + bm (shared by every layer); fin = Wf SiLU(temb) + bf
 *   x = [latent Wp^T + bp ; text]   image rows first, then text rows
 *   positions: image (n_txt, h, w), text (j, 0, 0); 3D RoPE on rope_axes
 *   n_layers x dit_block_forward
 *   v = (LN(x_img) (1 + fin.scale) + fin.shift) Wout^T + bout
 *   latent <- latent + (sigma_next - sigma) v
 * latent: device fp32 [grid_h grid_w, C], read and overwritten.
 * text:   device bf16 [n_txt, H].
 * velocity_out: device fp32 [grid_h grid_w, C] receiving v, or NULL. */
dit_status dit_denoise_step(const dit_model_config* cfg, const dit_model_weights* w,
                            float* latent, const void* text, int32_t grid_h,
                            int32_t grid_w, int32_t n_txt, float sigma,
                            float sigma_next, float* velocity_out, void* workspace,
                            size_t ws_bytes, void* stream);

/* Flow-matching Euler update x[i] <- x[i] + (sigma_next - sigma) v[i], the
 * product rounded before the add ([ZFLOW] section IV, sign +1).
 * x, v: device fp32 [n]. */
dit_status flowmatch_euler_step(float* x, const float* v, int64_t n, float sigma,
                                float sigma_next, void* stream);

/* Shifted flow-matching sigmas ([ERNIE] section I: FlowMatchEulerDiscrete,
 * shift 4.0, exponential time shift): s_i = 1 - i / n_steps and
 * sigma_i = shift s_i / (1 + (shift - 1) s_i), i = 0..n_steps, computed in
 * double and rounded to float.  out_host: HOST float [n_steps + 1]. */
dit_status flowmatch_sigmas(int32_t n_steps, float shift, float* out_host);

/* ------------------------------------------------- the path's stages, exposed
 * one by one so that each kernel can be checked on its own. */

/* y = x W^T with a fused epilogue.  a: device bf16 [M, K] (row stride lda
 * elements); w: device bf16 [N, K] (row stride ldw).  Epilogues:
 *   DIT_EPI_BF16:     out bf16 [M, N] (ldo)       out = y
 *   DIT_EPI_F32_BIAS: out fp32 [M, N] (ldo)       out = y + bias (bias may be NULL)
 *   DIT_EPI_RESIDUAL: out fp32 [M, N] (ldo)       out += gate * y  (gate [N] fp32,
 *                     NULL = 1) -- the gated residual ([ERNIE] section VII,
 *                     Decision 1)
 *   DIT_EPI_SWIGLU:   w holds [Wg; Wu] ([2F, K], gate rows first), N = F,
 *                     out bf16 [M, F] = SiLU(x Wg^T) * (x Wu^T)
 *   DIT_EPI_GEGLU, DIT_EPI_RESIDUAL_TANH, DIT_EPI_RESIDUAL_SIGMOID: the
 *                     variants of the two above (see the enum) */
enum {
  DIT_EPI_BF16 = 0, DIT_EPI_F32_BIAS = 1, DIT_EPI_RESIDUAL = 2, DIT_EPI_SWIGLU = 3,
  DIT_EPI_GEGLU = 4,             /* as SWIGLU with the clamped tanh GELU */
  DIT_EPI_RESIDUAL_TANH = 5,     /* out += tanh(gate) * y */
  DIT_EPI_RESIDUAL_SIGMOID = 6   /* out += sigmoid(gate) * y */
};
dit_status dit_linear(int32_t epilogue, const void* a, int64_t lda, const void* w,
                      int64_t ldw, int32_t M, int32_t N, int32_t K, void* out,
                      int64_t ldo, const float* bias_or_gate, void* stream);

/* The QKV projection with its fused epilogue ([ERNIE] section IV; [ZFLOW]
 * section VI, the fused per-head norm then rotation): [q|k|v] = a Wqkv^T, then per head
 * q <- RoPE(LN_d(q) q_g + q_b), k likewise, v unchanged.
 * a: device bf16 [n_tokens, H].  Outputs:
 *   qk: device bf16 [n_heads + n_kv_heads][n_tokens][d], head-major: q heads
 *       then k heads, each head's rows contiguous
 *   vt: device bf16 [n_seqs, n_kv_heads, d, s_pad], v transposed per sequence,
 *       s_pad = round_up(n_tokens / n_seqs, 8); columns >= seq length unused.
 * rope_cos, rope_sin: pair-major tables as for dit_block_forward. */
dit_status dit_qkv_rope(const dit_block_config* cfg, const dit_block_weights* w,
                        const void* a, int32_t n_tokens, int32_t n_seqs,
                        const float* rope_cos, const float* rope_sin, void* qk,
                        void* vt, void* stream);

/* dit_qkv_rope in the W8A8 format (cfg->linear_format == 1): a holds e4m3
 * codes [n_tokens, H] of the rotated normed rows (dit_ln_modulate_rotate_
 * quantize) with row scales a_scales [n_tokens]; w->w_qkv holds the rotated
 * weight's codes and w->w_qkv_scale their row scales.  Outputs as
 * dit_qkv_rope. */
dit_status dit_qkv_rope_e4m3(const dit_block_config* cfg, const dit_block_weights* w,
                             const void* a, const float* a_scales, int32_t n_tokens,
                             int32_t n_seqs, const float* rope_cos, const float* rope_sin,
                             void* qk, void* vt, void* stream);

/* Non-causal attention per sequence ([ERNIE] section VII, Decision 2: no
 * mask) with grouped KV heads ([ZFLOW] section VI, attention(heads,
 * kv_heads)): o_h = softmax(q_h k_g^T / sqrt(d)) v_g, g = h / (n_heads /
 * n_kv_heads).  qk, vt as written by dit_qkv_rope; o: device bf16
 * [n_tokens, n_heads d]. */
dit_status dit_attention(const dit_block_config* cfg, const void* qk, const void* vt,
                         int32_t n_tokens, int32_t n_seqs, void* o, void* stream);

/* Norm over each row of x then
 *   mode 0 (AdaLN): out = n (1 + p1) + p0   (p0 = shift, p1 = scale)
 *   mode 1 (affine): out = n p0 + p1         (p0 = gain, p1 = bias)
 * with n = LayerNorm(x) (biased variance, eps); add 2 to the mode for
 * n = RMSNorm(x) = x / sqrt(mean(x^2) + eps) ([ERNIE] section IV).
 * x: device fp32 [rows, H] (row stride ldx); out: device bf16 [rows, H]. */
dit_status dit_ln_modulate(int32_t mode, const float* x, int64_t ldx, int32_t rows,
                           int32_t H, const float* p0, const float* p1, float eps,
                           void* out, void* stream);

/* W8A8 coding of the rows of a bf16 matrix ([ZFLOW] section VII: 8-bit codes
 * per row, H256 rotation on both sides, exact in real arithmetic because
 * (x H)(W H)^T = x W^T for orthogonal H).  Each row is multiplied, in
 * independent blocks of 256 columns, by the 256-point Sylvester Hadamard
 * matrix scaled by 1/16 (the fast Walsh-Hadamard transform in fp32); then
 * amax = max |y|, scales[r] = amax / 448 and codes = e4m3(y * (448 / amax)),
 * rounded to nearest even and saturated (an all-zero row: scale 0, codes 0).
 * Used offline on the weights and, inside the block, on the activations.
 * x: device bf16 [rows, K] (row stride ldx elements); K a multiple of 256,
 * at most 16384.  codes: device bytes [rows, K] (row stride ldq bytes, a
 * multiple of 16); scales: device fp32 [rows]. */
dit_status dit_rotate_quantize(const void* x, int64_t ldx, int32_t rows, int32_t K,
                               void* codes, int64_t ldq, float* scales, void* stream);

/* dit_ln_modulate's row (same modes) rotated and coded as dit_rotate_quantize
 * does, without writing it in bf16: the A operand of the QKV and gate/up
 * projections in the W8A8 format.  H a multiple of 256, at most 8192.
 * codes: device bytes [rows, H] (row stride ldq); scales: device fp32 [rows]. */
dit_status dit_ln_modulate_rotate_quantize(int32_t mode, const float* x, int64_t ldx,
                                           int32_t rows, int32_t H, const float* p0,
                                           const float* p1, float eps, void* codes,
                                           int64_t ldq, float* scales, void* stream);

/* dit_linear on e4m3 codes: y[i, n] = a_scales[i] w_scales[n] sum_k a[i, k]
 * w[n, k], accumulated in fp32 on the tensor cores, then the same epilogues
 * as dit_linear.  a: device e4m3 [M, K] (row stride lda bytes), a_scales
 * [M]; w: device e4m3 [N, K] (ldw bytes; [2F, K] for the GLU epilogues),
 * w_scales [N] ([2F]).  K a multiple of 16. */
dit_status dit_linear_e4m3(int32_t epilogue, const void* a, const float* a_scales,
                           int64_t lda, const void* w, const float* w_scales, int64_t ldw,
                           int32_t M, int32_t N, int32_t K, void* out, int64_t ldo,
                           const float* bias_or_gate, void* stream);

/* Timestep conditioning of one step ([ZFLOW] section IV: flip_sin_to_cos
 * sinusoid; [ERNIE] section IV, adaLN split and section V, Bug 4, final
 * chunk order): writes mod [6H] and fin [2H] (device fp32).  scratch: device
 * fp32 [t_dim + 2H]. */
dit_status dit_timestep_conditioning(const dit_model_config* cfg,
                                     const dit_model_weights* w, float sigma,
                                     float* mod, float* fin, float* scratch,
                                     void* stream);

/* The same timestep conditioning for callers that cannot allocate device
 * memory: it needs no scratch argument.  No counterpart on the pages; this is
 * an interface addition of this library.
 *
 * Who needs it: code that is handed a stream but may not allocate on it --
 * a host application or inference server that gives this library a fixed
 * memory budget and forbids allocations behind its back, or a caller on a
 * latency-critical path where cudaMalloc/cudaFree would synchronise the
 * device.  The scratch (t_dim + 2 * hidden floats) is a static array inside
 * libdit.so of 32768 floats (128 KiB), held on every GPU that loads the
 * library until the process exits.
 *
 * Limits and behaviour:
 *   - t_dim + 2 * hidden > 32768 returns DIT_EUNSUPPORTED (nothing enqueued).
 *     Within the model limits (t_dim <= 16384, hidden <= 8192) the scratch
 *     always suffices; t_dim > 16384 returns DIT_EUNSUPPORTED, as it does
 *     for every call that takes a dit_model_config.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - The first call on a device asks the runtime for the array's device
 *     address (once per device, that device current); make that first call
 *     before any stream capture.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents; every word is written before it is read, so no clearing is
 *     needed.  Calls that overlap on the GPU (different streams, or
 *     concurrent host threads) race on it: serialise them.
 * mod [6H] and fin [2H]: device fp32 outputs, as dit_timestep_conditioning. */
dit_status dit_timestep_conditioning_noalloc(const dit_model_config* cfg,
                                             const dit_model_weights* w, float sigma,
                                             float* mod, float* fin, void* stream);

/* RoPE tables for the joint DiT sequence ([ERNIE] section IV token layout and
 * section VII, Decision 3): token t < grid_h grid_w is image cell
 * (t / grid_w, t % grid_w) at position (n_txt, h, w); token t >= grid_h grid_w
 * is text token j = t - grid_h grid_w at (j, 0, 0).  Pair k of axis a (the
 * head vector split into consecutive chunks of rope_axes[a]) turns by
 * pos_a theta^(-2k / rope_axes[a]).  cos, sin: device fp32 [d/2, N]
 * (pair-major: entry (k, t) at k N + t), N = grid_h grid_w + n_txt. */
dit_status dit_rope_table_grid(int32_t grid_h, int32_t grid_w, int32_t n_txt,
                               const int32_t* rope_axes, float theta, float* cos_out,
                               float* sin_out, void* stream);

/* Same from explicit positions: pos device int32 [n, 3]; cos, sin [d/2, n]. */
dit_status dit_rope_table_pos(const int32_t* pos, int32_t n, const int32_t* rope_axes,
                              float theta, float* cos_out, float* sin_out, void* stream);

/* Rotate-half RoPE tables of the pre-norm ViT ([MAKEPAD]: rotate-half rope
 * from tables): n_prefix unrotated tokens, then patch (r, c) of a grid_h x
 * grid_w grid; pair k < d/4 turns by r w_k, pair d/4 <= k < d/2 by
 * c w_(k - d/4), w_k = base^(-k / (d/4)).  cos, sin: device fp32
 * [d/2, n_prefix + grid_h grid_w] (pair-major). */
dit_status dit_rope_table_vit(int32_t grid_h, int32_t grid_w, int32_t n_prefix,
                              int32_t head_dim, float base, float* cos_out,
                              float* sin_out, void* stream);

/* ------------------------------------------------------------- diagnostics */

/* Reads and clears the device error word of the current device (synchronises
 * `stream`).  DIT_ETIMEOUT if a bounded wait inside a kernel ran out since
 * the last call, DIT_ECUDA on a CUDA error, else DIT_OK. */
dit_status dit_last_device_error(void* stream);

/* Limit, in nanoseconds, of every bounded wait inside the kernels of the
 * current device (default 2e9).  Tests shorten it to exercise the timeout. */
dit_status dit_set_wait_timeout_ns(uint64_t ns);

/* Launches one kernel that waits on a barrier nothing will complete, so that
 * its bounded wait runs out and sets the error word.  Exercises the failure
 * path without a fault; used by the tests. */
dit_status dit_debug_stuck_wait(void* stream);

/* Kernels launched by the library on this thread since the last reset
 * (host-side launch counter; reset when `reset` is non-zero). */
int64_t dit_launch_count(int32_t reset);

const char* dit_status_string(dit_status s);

#ifdef __cplusplus
}
#endif
#endif /* DIT_H_ */
