/* gpt2.h - C ABI of libgpt2.so: one GPT-2 pretraining step on one B300 (sm_103a).
 *
 * What the step computes (the pages this follows, by title and section):
 *   - token + position embedding, pre-LN blocks (LayerNorm -> QKV -> causal
 *     softmax attention -> projection + residual -> LayerNorm -> 4C GELU MLP +
 *     residual), final LayerNorm, lm_head tied to wte over a vocabulary padded
 *     50257 -> 50304, mean cross-entropy over all B*T positions:
 *     "Let's reproduce GPT-2 (124M)" wiki page, "Training recipe details"
 *     (weight tying, 1/sqrt(2N) residual init) and "GPU optimisation ladder"
 *     (FlashAttention, vocab padding); qntz.me nanoGPT page (block contents,
 *     init loss ln V); llm.c 1558M article run log (parameter layout, bf16
 *     params/grads with fp32 master weights and AdamW state);
 *   - global-norm gradient clip and AdamW(beta1, beta2, eps) with decoupled weight
 *     decay on the 2-D matrices only: wiki page "Training recipe details";
 *     llm.c article "Parameter guide" (-c 0.1 decays 2-D weights only).
 *
 * Conventions for every call:
 *   - Pointers named d_* or documented as device pointers are CUDA device
 *     addresses; h_* are host addresses.  The library never allocates device
 *     memory: the caller owns the arena and all I/O buffers.
 *   - All GPU work is enqueued on the caller's stream (a cudaStream_t passed
 *     as void*; NULL = legacy default stream).  Calls do not synchronise except
 *     where a host output (h_loss, h_norm, gpt2_get_tensor to host,
 *     gpt2_sync_status) is requested.
 *   - Every function returns GPT2_OK (0) or a negative status below; shape and
 *     pointer errors are detected on the host before anything is enqueued.
 *   - Results are bitwise reproducible run to run on the same device.
 *
 * Parameter order (canonical flat fp32 vector, Linear weights [out, in]):
 *   wte[Vpad,C] wpe[T,C] ln1w[L,C] ln1b[L,C] qkvw[L,3C,C] qkvb[L,3C]
 *   attprojw[L,C,C] attprojb[L,C] ln2w[L,C] ln2b[L,C] fcw[L,4C,C] fcb[L,4C]
 *   fcprojw[L,C,4C] fcprojb[L,C] lnfw[C] lnfb[C]
 *   total N = Vpad*C + T*C + L*(12C^2 + 13C) + 2C  (1557686400 for L=48, C=1600,
 *   Vpad=50304, T=1024, as printed in the llm.c 1558M run log).
 */
#ifndef GPT2_B300_H
#define GPT2_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum gpt2_status {
  GPT2_OK = 0,
  GPT2_E_INVAL = -1,      /* bad shape, size, alignment or null pointer */
  GPT2_E_STATE = -2,      /* call out of order (forward -> backward -> clip_adamw) */
  GPT2_E_TOKEN = -3,      /* a token or target id was outside [0, V); it was clamped to 0 */
  GPT2_E_CUDA = -4,       /* a CUDA runtime call failed (see gpt2_last_cuda_error) */
  GPT2_E_TIMEOUT = -5,    /* a bounded wait inside a pipelined kernel expired */
  GPT2_E_NONFINITE = -6,  /* the loss or the gradient norm is not finite */
  GPT2_E_UNSUPPORTED = -7 /* shape valid but outside what this build handles */
};

enum gpt2_precision {
  GPT2_FP32 = 0, /* fp32 params, activations and grads; CUDA-core GEMMs (parity mode) */
  GPT2_BF16 = 1  /* bf16 params/activations/grads, fp32 master + AdamW state; tcgen05 GEMMs */
};

enum gpt2_tensor {
  GPT2_PARAMS = 0, /* working parameters (bf16 in GPT2_BF16 mode) */
  GPT2_GRADS = 1,  /* parameter gradients of the last backward */
  GPT2_ADAM_M = 2, /* AdamW first moment (fp32) */
  GPT2_ADAM_V = 3, /* AdamW second moment (fp32) */
  GPT2_MASTER = 4, /* fp32 master weights (same as PARAMS in GPT2_FP32 mode) */
  GPT2_GRAD_ACC = 5 /* fp32 gradient accumulator of gpt2_grad_accumulate */
};

/* Kernel classes of the per-region timing (gpt2_profile). */
enum gpt2_kernel_class {
  GPT2_K_GEMM = 0,      /* every Linear incl. the fused classifier logits (tensor cores) */
  GPT2_K_SPLITK = 1,    /* fp32 split-K reduction of the many-split weight-gradient GEMMs */
  GPT2_K_ATTN_FWD = 2,  /* fused causal attention forward */
  GPT2_K_ATTN_BWD = 3,  /* rowsum(dO*O) + dK/dV + dQ kernels */
  GPT2_K_LN_FWD = 4,
  GPT2_K_LN_BWD = 5,    /* incl. the fixed-order dgamma/dbeta reduction */
  GPT2_K_CE = 6,        /* statistics merge, mean loss, dlogits in place */
  GPT2_K_ENCODER = 7,   /* id checks + gather (forward), sort + scatter (backward) */
  GPT2_K_BIAS_GRAD = 8, /* bias gradients (column sums) */
  GPT2_K_NORM = 9,      /* global gradient norm */
  GPT2_K_ADAMW = 10,    /* fused clip + AdamW + bf16 copy */
  GPT2_K_RECOMPUTE = 11, /* activation recompute in the backward (gelu(h), LayerNorm outputs) */
  GPT2_K_COUNT = 12
};

typedef struct gpt2 gpt2_t;

/* Number of parameters N (canonical order above). */
size_t gpt2_num_params(int L, int C, int Vpad, int T);

/* Bytes of device memory gpt2_create needs for this shape (B = sequences per
 * step, T = sequence length = number of positions in wpe).  Constant for the
 * life of the handle: nothing is allocated afterwards. 0 on invalid shape. */
size_t gpt2_arena_bytes(int L, int H, int C, int V, int Vpad, int T, int B, int precision);

/* Create a step driver over a caller-owned device arena of >= gpt2_arena_bytes
 * bytes (256-byte aligned).  Requirements: C % H == 0, C % 8 == 0, Vpad >= V,
 * Vpad % 8 == 0, B*T <= 16384; GPT2_BF16 additionally needs head size C/H == 64
 * and C <= 2048; GPT2_FP32 needs C/H <= 128 and C <= 1024.  Parameters start
 * at zero: call gpt2_set_params before the first step. */
int gpt2_create(int L, int H, int C, int V, int Vpad, int T, int B, int precision, void* d_arena,
                size_t arena_bytes, void* stream, gpt2_t** out);
void gpt2_destroy(gpt2_t* h);
int gpt2_set_stream(gpt2_t* h, void* stream);

/* Activation recompute (llm.c GPT-2 1558M article, "Parameter guide" and
 * "Memory guide": -r 1 recomputes GELU in the backward pass instead of keeping
 * it, -r 2 also recomputes LayerNorm; compute traded for memory).  gpt2_create
 * and gpt2_arena_bytes are these calls with recompute = 0 (everything kept):
 *   1  the forward keeps h = x W_fc^T + b per layer and gelu(h) only until the
 *      projection GEMM has read it; the backward recomputes gelu(h) (for the
 *      projection's weight gradient) and gelu'(h) (in the GELU' epilogue) from
 *      h.  Saves (L - 1) * B*T * 4C storage elements.
 *   2  as 1, and the LayerNorm outputs ln1 / ln2 are not kept either: the
 *      backward recomputes each from the stored residual (the same kernel, so
 *      the same bits) right before the weight-gradient GEMM that reads it.
 *      Saves another (2L - 1) * B*T * C elements.
 * Results agree with recompute = 0 within the bf16 tolerances (the recomputed
 * GELU uses the rounded h); other values are GPT2_E_INVAL. */
size_t gpt2_arena_bytes_r(int L, int H, int C, int V, int Vpad, int T, int B, int precision, int recompute);
int gpt2_create_r(int L, int H, int C, int V, int Vpad, int T, int B, int precision, int recompute, void* d_arena,
                  size_t arena_bytes, void* stream, gpt2_t** out);

/* Load N fp32 parameters (canonical order) from host (on_device = 0) or device
 * memory; in GPT2_BF16 mode they become the fp32 master copy and the working
 * bf16 copy is their round-to-nearest-even.  Zeroes the AdamW moments. */
int gpt2_set_params(gpt2_t* h, const float* params, int on_device);

/* Copy one state tensor (enum gpt2_tensor) as N fp32 values to dst (host or device). */
int gpt2_get_tensor(gpt2_t* h, int which, float* dst, int dst_on_device);

/* Forward pass and loss.  d_tokens / d_targets: device int32 [B, T] (copied
 * into the arena, so they may be reused after the call is enqueued).  The
 * fused classifier also turns the logits into dlogits in place, so the next
 * gpt2_backward needs no other input.  The mean loss lands in device memory
 * (gpt2_device_loss); h_loss, if not NULL, receives it after a stream sync,
 * and then a clamped token id is reported as GPT2_E_TOKEN. */
int gpt2_forward(gpt2_t* h, const int32_t* d_tokens, const int32_t* d_targets, float* h_loss);

/* Backward pass of the last forward: writes every parameter gradient. */
int gpt2_backward(gpt2_t* h);

/* Global-norm clip to max_norm (scale = max_norm / norm when norm > max_norm)
 * followed by AdamW at step t (step_t >= 1; step_t = 0 takes t from a device
 * counter that each call increments and gpt2_set_params resets, so a CUDA
 * graph of the step stays correct across replays): m = b1 m + (1-b1) g, v = b2 v + (1-b2) g^2,
 * w -= lr (m/(1-b1^t) / (sqrt(v/(1-b2^t)) + eps) + weight_decay * w) with the
 * decay applied to wte, wpe, qkvw, attprojw, fcw, fcprojw only.  The norm
 * stays on the device; h_norm, if not NULL, receives it after a stream sync. */
int gpt2_clip_adamw(gpt2_t* h, float lr, float beta1, float beta2, float eps, float weight_decay,
                    float max_norm, int step_t, float* h_norm);

/* Gradient accumulation over micro-batches (llm.c GPT-2 1558M article: the
 * total batch of -d tokens is reached in micro-steps of B*T; its run log sets
 * grad_accum_steps=8).  Call after gpt2_backward: acc = (first ? 0 : acc) +
 * scale * grads, in fp32 (scale = 1/k for k micro-batches of B*T positions, so
 * acc is the gradient of the mean loss over all of them).  gpt2_forward and
 * gpt2_backward may then run on the next micro-batch.  gpt2_clip_adamw_accumulated
 * is gpt2_clip_adamw with acc as the gradient (norm, clip and AdamW over it).
 * Call order is checked (GPT2_E_STATE). */
int gpt2_grad_accumulate(gpt2_t* h, int first, float scale);
int gpt2_clip_adamw_accumulated(gpt2_t* h, float lr, float beta1, float beta2, float eps,
                                float weight_decay, float max_norm, int step_t, float* h_norm);

/* Learning rate of step step_t (1-based, like step_t above) under linear warmup
 * then cosine decay (llm.c GPT-2 1558M article, "Parameter guide": -k cosine,
 * -u warmup, -q final fraction, -x total steps; the run log prints the warmup
 * values): max_lr * t / warmup_steps for t <= warmup_steps; then
 * max_lr * (f + (1 - f) * (1 + cos(pi * r)) / 2) with f = final_frac and
 * r = (t - 1 - warmup_steps) / (total_steps - warmup_steps) clamped to [0, 1].
 * Host only (no device work).  Returns a negative value for invalid arguments
 * (t < 1, warmup_steps < 0, total_steps <= warmup_steps, max_lr < 0). */
float gpt2_lr_schedule(int step_t, float max_lr, int warmup_steps, int total_steps, float final_frac);

/* One whole step from host buffers: copies h_tokens / h_targets (int32 [B, T])
 * to the device, runs forward, backward, clip + AdamW, and copies the loss and
 * gradient norm back (h_loss / h_norm may be NULL).  Synchronises the stream.
 * The first call captures the step as one CUDA graph (on a private stream, with
 * pinned staging buffers for tokens, targets, hyperparameters and the results)
 * and every call replays it on the handle's stream, so the arguments may change
 * from call to call; while gpt2_profile is on the step runs eagerly instead.
 * Returns GPT2_E_TOKEN / GPT2_E_TIMEOUT / GPT2_E_NONFINITE for this step's
 * status bits (which it clears). */
int gpt2_train_step_host(gpt2_t* h, const int32_t* h_tokens, const int32_t* h_targets, float lr,
                         float beta1, float beta2, float eps, float weight_decay, float max_norm,
                         int step_t, float* h_loss, float* h_norm);

/* Device addresses of the last loss (fp32) and of {norm, clip scale} (fp32[2]). */
const float* gpt2_device_loss(gpt2_t* h);
const float* gpt2_device_norm(gpt2_t* h);

/* Per-region timing: while on, every kernel group the step issues is bracketed
 * by CUDA events on the stream (do not capture a graph while it is on).  `on`
 * clears earlier records.  gpt2_profile_read synchronises and returns, for one
 * enum gpt2_kernel_class, the number of regions, their summed milliseconds and
 * their summed algorithmic flops and bytes. */
int gpt2_profile(gpt2_t* h, int on);
int gpt2_profile_read(gpt2_t* h, int kernel_class, int* regions, double* ms, double* flops,
                      double* bytes);
/* The recorded regions one by one (in issue order): count, then region i's
 * class, dims (GEMM regions: M, N, K, A MN-major, B MN-major, epilogue kind;
 * zeros otherwise; int[6]), milliseconds, flops and bytes. */
int gpt2_profile_regions(gpt2_t* h);
int gpt2_profile_region(gpt2_t* h, int i, int* kernel_class, int* dims, double* ms, double* flops,
                        double* bytes);

/* Synchronise the stream, read and clear the device status word; returns
 * GPT2_OK, GPT2_E_TOKEN, GPT2_E_TIMEOUT or GPT2_E_NONFINITE. */
int gpt2_sync_status(gpt2_t* h);

/* Update guard (llm.c GPT-2 1558M article, "400B token run": once instabilities
 * appeared, the run skipped the parameter update whenever it detected a
 * momentary spike, flags -sl 5.0 -sg 5.0; its run log prints a z-score beside
 * the loss and the norm, shown as "+nan" until enough steps have passed).
 * Every gpt2_clip_adamw / gpt2_clip_adamw_accumulated, on the device:
 *   - scores the step's mean loss (for the accumulated call: the scale-weighted
 *     sum of the micro-batch losses) and its gradient norm against the last
 *     `window` finite values of each: z = (x - mean) / std with the population
 *     mean and standard deviation; z is NaN while fewer than `window` values are
 *     held, and 0 (or +-inf) when the deviation is 0;
 *   - skips the update, leaving master weights, working weights, m and v
 *     untouched and the device step counter where it was, when the loss or the
 *     norm is not finite (always; the call reports GPT2_E_NONFINITE as before),
 *     or when loss_z > 0 and the loss's z exceeds it, or norm_z > 0 and the
 *     norm's z exceeds it (a spike: the call returns GPT2_OK);
 *   - then adds the step's loss and norm to the window if both are finite.
 * gpt2_set_guard sets the thresholds (<= 0 turns a check off) and the window
 * (2 .. 256) and empties the window and the counters; it synchronises the
 * stream.  A new handle starts with both checks off and a window of 128.
 * gpt2_set_params does not touch the guard.  gpt2_guard_read synchronises and
 * returns the last step's z-scores, the numbers of updates skipped for a spike
 * and for a non-finite value, and whether the last update was skipped (any
 * pointer may be NULL). */
int gpt2_set_guard(gpt2_t* h, float loss_z, float norm_z, int window);
int gpt2_guard_read(gpt2_t* h, float* z_loss, float* z_norm, int* skipped_spike, int* skipped_nonfinite,
                    int* last_skipped);

const char* gpt2_strerror(int status);
/* Text of the last CUDA error seen by any call in this process. */
const char* gpt2_last_cuda_error(void);

/* ---------------------------------------------------------------- standalone kernels
 * Causal attention over bf16 tensors, head size d = 64, fp32 accumulation,
 * softmax scale `scale` ("Let's reproduce GPT-2 (124M)" wiki page, "GPU
 * optimisation ladder": FlashAttention computes the exact causal softmax
 * attention without materialising the T x T matrix, 7.6x faster).  Element (b, h, t, i) of q, k, v, dq, dk, dv is at
 * b*sb + h*sh + t*st + i; of o and dO at b*osb + h*osh + t*ost + i (elements;
 * all strides multiples of 8, pointers 16-byte aligned).  lse: fp32 [B, H, T],
 * natural-log sum of exp of the scaled, masked scores (keys j <= query t).
 * The T x T matrix is never stored. */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int T,
             int d, long long sb, long long sh, long long st, long long osb, long long osh,
             long long ost, float scale, void* stream);
/* Gradients of attn_fwd (same page and section: the backward of the exact
 * attention, dV = P^T dO, dP = dO V^T, dS = P o (dP - rowsum(dO o O)),
 * dQ = scale dS K, dK = scale dS^T Q, recomputing P from lse).  Tensor layouts
 * as attn_fwd; dq, dk, dv are written (not accumulated).  workspace: device,
 * >= attn_workspace_bytes(B, H, T) bytes, 16-byte aligned, owned by the caller
 * and free again when the call's kernels have run. */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dO, void* dq, void* dk, void* dv, int B, int H, int T, int d, long long sb,
             long long sh, long long st, long long osb, long long osh, long long ost, float scale,
             void* workspace, size_t workspace_bytes, void* stream);
size_t attn_workspace_bytes(int B, int H, int T);

/* attn_bwd for callers that cannot allocate device memory; the pages have no
 * counterpart of this call.  Some callers cannot hand the library a workspace:
 * a host runtime that gives the whole device to its own memory pool and
 * forbids library allocations, or a latency-critical loop that cannot afford
 * cudaMalloc's implicit device synchronisation.  This call takes the same
 * arguments as attn_bwd minus the workspace, computes the same gradients with
 * the same kernels, and allocates nothing: its scratch (fp32 rowsum(dO * O),
 * one float per (b, h, t)) is a fixed array in the library's static device
 * memory, ATTN_BWD_NOALLOC_MAX_ROWS floats (4 MiB), which every GPU that
 * loads the library holds until the process exits.
 *   - B * H * T > ATTN_BWD_NOALLOC_MAX_ROWS returns GPT2_E_UNSUPPORTED before
 *     anything is enqueued; other argument errors are those of attn_bwd.
 *   - The first call on a device, made with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress) and caches it with the id
 *     of the current context; make that first call before any stream capture.
 *     After a device reset the first call in the new context looks it up again.
 *     A failed lookup returns GPT2_E_CUDA (text in gpt2_last_cuda_error).
 *   - Every call on a device shares the one array.  Calls whose kernels may
 *     overlap on the GPU (different streams with no ordering) race on it.  The
 *     array keeps the last call's contents; nothing needs clearing, since
 *     every row is written before it is read. */
#define ATTN_BWD_NOALLOC_MAX_ROWS 1048576
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dO, void* dq, void* dk, void* dv, int B, int H, int T, int d,
                     long long sb, long long sh, long long st, long long osb, long long osh,
                     long long ost, float scale, void* stream);

/* Tied lm_head + mean cross-entropy, fused ("Let's reproduce GPT-2 (124M)"
 * wiki page, "Training recipe details": lm_head shares wte; "GPU optimisation
 * ladder": the vocabulary padded 50257 -> 50304; qntz.me nanoGPT page: the
 * loss is the mean cross-entropy, ln V at a uniform init): logits = x w^T (x bf16 [M, C],
 * w bf16 [Vpad, C]; columns >= V excluded from the softmax), loss = mean over
 * rows of lse - logit[target]; then dlogits = (softmax - onehot) / M,
 * dx = dlogits w (bf16 [M, C]) and dw = dlogits^T x (bf16 [Vpad, C], pad rows 0).
 * d_loss: device fp32 scalar.  targets: device int32 [M] in [0, V).
 * workspace >= classifier_workspace_bytes(M, C, Vpad) (holds the bf16 logits). */
int classifier_fwd_bwd(const void* x, const void* w, const int32_t* targets, int M, int C, int V,
                       int Vpad, float* d_loss, void* dx, void* dw, void* workspace,
                       size_t workspace_bytes, void* stream);
size_t classifier_workspace_bytes(int M, int C, int Vpad);

/* Token + position embedding on its own (the gather of the forward pass):
 * x0[b, t, :] = wte[tok[b, t], :] + wpe[t, :] with one fp32 addition and one
 * rounding to the storage type (precision: GPT2_FP32 -> float, GPT2_BF16 -> bf16
 * tensors).  tok: device int32 [B, T]; ids outside [0, V) are clamped to 0 and
 * bit 0 of *d_status (device uint32, may be NULL) is set.  Bit-exact. */
int gpt2_encoder_fwd(const int32_t* tok, const void* wte, const void* wpe, void* x0, int B, int T,
                     int C, int V, int precision, void* d_status, void* stream);
/* The scatter of the backward pass.  For every vocab id v: the positions
 * holding v, in ascending order, are cut into runs of 64; each run's dx0 rows
 * (fp32 [B, T, C]) are summed from zero in ascending order, the run sums are
 * added in run order from zero, and dwte[v] = dwte[v] + total (one rounding).
 * dwpe[t] = sum over b ascending of dx0[b, t] (written, not accumulated).
 * dx0 is consumed: rows of it are overwritten with run sums.  workspace >=
 * 8*B*T bytes.  Bit-exact and deterministic. */
int gpt2_encoder_bwd(const int32_t* tok, float* dx0, void* dwte, void* dwpe, int B, int T, int C,
                     int V, int precision, void* workspace, size_t workspace_bytes, void* stream);

/* The tensor-core GEMM engine on its own (bf16 in, fp32 accumulate):
 * D[m, n] = sum_k A(m, k) B(n, k), A(m, k) = A[m*lda + k] (a_mn = 0) or
 * A[k*lda + m] (a_mn = 1), likewise B(n, k) with b_mn; D bf16 (d_f32 = 0) or
 * fp32 (d_f32 = 1) with leading dimension ldd.  N, lda, ldb, ldd multiples of 8.
 * splits > 1 divides K and needs workspace >= splits*M*N*4 bytes (0 = choose).
 * splits = -1 picks a schedule that adds partial sums inside the kernel where
 * it pays: stream-K (whole waves of output tiles as usual, the leftover tiles
 * of a part-empty last wave cut evenly along K over all SMs) for tiles deep in
 * K, or K splits finished by the last split when there are fewer tiles than
 * SMs; the sums are added in a fixed order (deterministic).  -2 takes stream-K
 * whenever the tiles do not fill whole waves.  Both need a 16-byte aligned
 * workspace of >= gemm_bf16_sk_workspace_bytes() bytes whose contents are zero
 * before its first use; every completed call leaves it reusable (a call whose
 * bounded waits expired may not: zero it again).  Calls that share a workspace
 * must not run concurrently.  The step driver lowers its own workspace's flags
 * whenever it reports GPT2_E_TIMEOUT. */
int gemm_bf16(const void* A, const void* B, void* D, int M, int N, int K, long long lda,
              long long ldb, long long ldd, int a_mn, int b_mn, int d_f32, int splits,
              void* workspace, size_t workspace_bytes, void* stream);
/* Workspace bytes of the splits = -1 / -2 schedules on the current device. */
size_t gemm_bf16_sk_workspace_bytes(void);
/* Number of CTA pairs (clusters of two CTAs on two SMs) the GEMM engine keeps
 * resident on the current device: its persistent grid is twice this. */
int gemm_bf16_pairs(void);

/* The GEMM engine with one of its fused epilogues, for tests.  As gemm_bf16
 * (bf16 D, same splits / workspace rules, no split > 1 with a fused epilogue)
 * with epi: 1 D = acc + bias[n]; 2 D = acc + bias[n] + X[m, n]; 3 h = acc +
 * bias[n], D = gelu'(h), D2 = gelu(h) (tanh form); 4 D = acc * X[m, n] and, if
 * colpart is not NULL, colpart[(m / 32) * N + n] = the fp32 sum of D over rows
 * m .. m + 31 before rounding.  bias: bf16 [N]; X, D2: bf16 [M, N] with leading
 * dimension ldd; colpart: fp32, ceil(M / 32) * N. */
int gemm_bf16_epilogue(const void* A, const void* B, void* D, void* D2, const void* bias, const void* X,
                       float* colpart, int M, int N, int K, long long lda, long long ldb, long long ldd,
                       int a_mn, int b_mn, int epi, int splits, void* workspace, size_t workspace_bytes,
                       void* stream);

/* Test hooks for the bounded waits (the pages have no counterpart).  Every
 * spin-wait in the pipelined kernels gives up after about 2 s, latches
 * GPT2_E_TIMEOUT in the call's status word and lets the kernel drain its copies,
 * free its tensor memory and return, so the context stays usable.  While a bit
 * of the mask is set, the launches that read it make one producer skip one
 * transfer, so the matching consumer's wait runs out:
 *   1  GEMM: the TMA producer skips its first shared-memory stage;
 *   2  GEMM stream-K / in-kernel split schedules: partial units never raise their
 *      ready flags, so the finishing CTAs' flag waits run out;
 *   4  attention forward: the producer skips its first K/V stage;
 *   8  attention backward, dQ kernel: the producer skips its first K/V stage;
 *  16  attention backward, dK/dV kernel: the producer skips its first Q/dO stage;
 *  32  streaming LayerNorm backward (bf16): one warp's first row copy is skipped.
 * gpt2_test_set_poison sets the whole mask and returns the previous one;
 * gpt2_test_set_gemm_poison(on) sets or clears bit 1 alone and returns its old
 * value.  The mask is process-wide and read at launch time: use it from one
 * thread with no other launches in flight. */
int gpt2_test_set_poison(int mask);
int gpt2_test_set_gemm_poison(int on);
/* One GEMM like gemm_bf16 (bf16 D, no fused epilogue) with a caller-owned
 * device status word (uint32, zeroed by the call), returning its status after a
 * stream sync: GPT2_OK or GPT2_E_TIMEOUT.  splits: 1 (plain) or -1 / -2 (the
 * in-kernel partial-sum schedules of gemm_bf16, with their workspace rules). */
int gemm_bf16_status(const void* A, const void* B, void* D, int M, int N, int K, long long lda,
                     long long ldb, long long ldd, int a_mn, int b_mn, int splits, void* workspace,
                     size_t workspace_bytes, void* d_status_word, void* stream);

#ifdef __cplusplus
}
#endif
#endif
