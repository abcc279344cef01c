// Host-side launchers of the GPT-2 step kernels (internal to libgpt2.so).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gpt2k {

// ------------------------------------------------------------------ host helpers (gpt2.cu)
// Records "where: <CUDA error text>" as this thread's last CUDA error (see
// gpt2_last_cuda_error) and returns GPT2_E_CUDA.
int cuda_fail(cudaError_t e, const char* where);
// Unique id of the CUDA context current on this thread, 0 when there is none.
// A device reset gives the device a new primary context with a new id, and
// with it new kernel attributes and new addresses of static device memory.
unsigned long long current_context_id();
// Per-device record of a one-time setting: the id of the context it was made in.
struct PerDeviceOnce {
  unsigned long long ctx[64] = {};
};
// Raises `kernel`'s dynamic shared-memory limit to `bytes` in the current
// context, once per device and context: the attribute belongs to the context,
// so a process that drives several GPUs (or resets one) sets it again there.
// Thread-safe.
cudaError_t smem_limit_once(const void* kernel, int bytes, PerDeviceOnce* once);

// Test hooks for the bounded waits (gpt2_test_set_poison): while a bit is set,
// the launches that read it make one producer skip one transfer, so that the
// matching consumer's bounded wait runs out.
enum PoisonBits {
  POISON_GEMM_TMA = 1,    // GEMM producer skips its first shared-memory stage
  POISON_GEMM_FLAG = 2,   // stream-K / split partial units never raise their ready flags
  POISON_ATTN_FWD = 4,    // attention forward producer skips its first K/V stage
  POISON_ATTN_DQ = 8,     // attention dQ kernel producer skips its first K/V stage
  POISON_ATTN_DKDV = 16,  // attention dK/dV kernel producer skips its first Q/dO stage
  POISON_LN_BWD = 32,     // streaming LayerNorm backward skips the first row copy of one warp
};
int test_poison();

// ------------------------------------------------------------------ GEMM
// D[m, n] = sum_k A(m, k) * B(n, k), fp32 accumulation, then an epilogue.
// A(m, k) = A[m * lda + k] when a_mn == 0 (K-major), A[k * lda + m] when 1.
// B(n, k) = B[n * ldb + k] when b_mn == 0 (K-major), B[k * ldb + n] when 1.
enum EpiKind {
  EPI_STORE = 0,       // D = acc                          (storage type)
  EPI_BIAS = 1,        // D = acc + bias[n]
  EPI_BIAS_RESID = 2,  // D = acc + bias[n] + resid[m, n]
  EPI_BIAS_GELU = 3,   // h = acc + bias[n];  D = gelu'(h), D2 = gelu(h)
  EPI_GELU_BWD = 4,    // D = acc * aux[m, n]  (aux = the gelu'(h) the forward stored)
  EPI_CE = 5,          // D = z = acc; per (row, N tile) max / sum exp over n < V; target logit
  EPI_F32 = 6,         // D (float*) = acc
  // activation recompute: the forward keeps only h, the backward derives gelu'(h) from it
  EPI_BIAS_GELU_H = 7, // h = round(acc + bias[n]);  D = h, D2 = gelu(h)
  EPI_GELU_BWD_H = 8,  // D = acc * gelu'(aux[m, n])  (aux = the h the forward stored)
};

struct GemmArgs {
  const void* A = nullptr; long long lda = 0; int a_mn = 0;
  const void* B = nullptr; long long ldb = 0; int b_mn = 0;
  int M = 0, N = 0, K = 0;
  int epi = EPI_STORE;
  void* D = nullptr; long long ldd = 0;
  const void* bias = nullptr;
  const void* resid = nullptr; long long ldr = 0;
  void* D2 = nullptr;
  const void* aux = nullptr; long long ldaux = 0;
  float* ce_max = nullptr; float* ce_sum = nullptr; int ce_ld = 0;
  float* ce_tgt = nullptr; const int32_t* targets = nullptr; int V = 0;
  // EPI_GELU_BWD / EPI_GELU_BWD_H, tcgen05 engine only: when set, colpart[(m / 32) * N + n] receives
  // the fp32 sum of D over rows m .. m + 31 (before rounding), ceil(M / 32) x N floats
  float* colpart = nullptr;
};

// bf16 operands on tcgen05 tensor cores (TMA -> smem ring -> MMA -> TMEM -> epilogue).
// `splits` > 1 splits K; partials go to `ws` as fp32 [splits][M][N] and a
// reduction kernel applies EPI_STORE / EPI_F32 (skipped when reduce == 0; the
// caller then runs splitk_reduce itself).
// `splits` == GEMM_TC_STREAM_K picks a schedule that adds partial sums inside
// the kernel where it pays (any epilogue): stream-K over the leftover tiles of
// a part-empty last wave when tiles are deep in K, or K splits finished by the
// last split when there are fewer tiles than SMs.  The partial sums are added
// in a fixed order (deterministic).  `ws` (>= gemm_tc_sk_ws_bytes(), 16-byte
// aligned) holds a flag area that must be zero before the first such call and
// is left zero by each call that completes, then the fp32 tile slots.  Calls
// sharing a `ws` must not overlap in time.  GEMM_TC_STREAM_K_FORCE takes
// stream-K whenever the tiles do not fill whole waves.  Returns 0 or a
// cudaError_t.
constexpr int GEMM_TC_STREAM_K = -1;
constexpr int GEMM_TC_STREAM_K_FORCE = -2;
// Where that schedule runs plain K splits with a separate reduction (more than
// two splits of a plain-store GEMM with fewer tiles than SMs) and reduce == 0,
// *reduce_splits receives the split count and the fp32 planes sit at
// ws + gemm_tc_sk_plane_offset(); the caller then runs splitk_reduce.
int gemm_tc(const GemmArgs& g, int splits, void* ws, size_t ws_bytes, unsigned* status,
            cudaStream_t s, int reduce = 1, int* reduce_splits = nullptr);
size_t gemm_tc_sk_plane_offset();
size_t gemm_tc_sk_ws_bytes();
// Splits the call above will actually use for this K (every split non-empty).
int gemm_tc_effective_splits(int K, int splits);
size_t gemm_tc_ws_bytes(int M, int N, int splits);
int gemm_tc_pick_splits(int M, int N, int K, int num_pairs);
// CTA pairs the engine runs on (resident at once on the current device).
int gemm_tc_pairs();
// Columns covered by one EPI_CE statistics partial (row m's partial j covers
// columns [j*cols, (j+1)*cols)).
int gemm_tc_stat_cols();
int num_sms();

// fp32 operands on CUDA cores (the fp32 parity mode).
int gemm_simt(const GemmArgs& g, cudaStream_t s);

// ------------------------------------------------------------------ attention
struct AttnArgs {
  const void *q = nullptr, *k = nullptr, *v = nullptr;
  void* o = nullptr; float* lse = nullptr;
  const void* dO = nullptr;
  void *dq = nullptr, *dk = nullptr, *dv = nullptr;
  float* Dbuf = nullptr;  // [B, H, T] rowsum(dO * O)
  int B = 0, H = 0, T = 0, d = 0;
  long long sb = 0, sh = 0, st = 0;     // q, k, v, dq, dk, dv (elements)
  long long osb = 0, osh = 0, ost = 0;  // o, dO
  float scale = 0.f;
  unsigned* status = nullptr;  // device status word for bounded-wait expiry (may be null)
  // tcgen05 backward only, may be null: bias_part[((b * nq + t / 128) * 4 + (t % 128) / 32) * 3C + c]
  // receives the fp32 sum over those 32 positions t of column c of [dq | dk | dv] (C = H * d,
  // nq = ceil(T / 128)), the partials of the QKV bias gradient
  float* bias_part = nullptr;
};
// Rows of AttnArgs::bias_part for batch B and sequence length T.
inline int attn_bias_part_rows(int B, int T) { return B * ((T + 127) / 128) * 4; }
// tcgen05 kernels (d = 64); a.status (may be null) receives ST_TIMEOUT on a bounded-wait expiry.
// attn_bwd_tc writes D = rowsum(dO * O) to a.Dbuf ([B, H, T] fp32 scratch) and uses it.
int attn_fwd_tc(const AttnArgs& a, cudaStream_t s);
int attn_bwd_tc(const AttnArgs& a, cudaStream_t s);
// bf16: attn_bwd_tc (stride checks first).
int attn_bwd_bf16(const AttnArgs& a, cudaStream_t s);
int attn_fwd_f32(const AttnArgs& a, cudaStream_t s);
int attn_bwd_f32(const AttnArgs& a, cudaStream_t s);

// ------------------------------------------------------------------ memory-bound
void check_ids(int32_t* ids, int n, int V, unsigned* status, cudaStream_t s);
template <typename T>
void encoder_fwd(T* x0, const int32_t* tok, const T* wte, const T* wpe, int B, int Tn, int C, int V,
                 unsigned* status, cudaStream_t s);
template <typename T>
void layernorm_fwd(T* y, float* mean, float* rstd, const T* x, const T* w, const T* b, int M, int C,
                   cudaStream_t s);
// dres (+)= LNbwd(dy); dres_b (optional) = storage copy of dres; dw, db = the LayerNorm's
// weight / bias gradients; dsum (optional) = column sum of the new dres.
// `status` (may be null) receives ST_TIMEOUT if a bounded wait of the streaming kernel expires.
template <typename T>
void layernorm_bwd(float* dres, T* dres_b, const T* dy, const T* x, const float* mean,
                   const float* rstd, const T* w, T* dw, T* db, T* dsum, float* partials, int M,
                   int C, int accumulate, cudaStream_t s, unsigned* status = nullptr);
size_t layernorm_bwd_partials_floats(int C);
template <typename T>
void colsum(T* out, const T* x, int M, int N, long long ld, float* partials, cudaStream_t s);
// out[n] = sum over p < nparts of partials[p * N + n], fixed order (deterministic).
template <typename T>
void colsum_reduce(T* out, const float* partials, int nparts, int N, cudaStream_t s);
size_t colsum_partials_floats(int N);
// y = gelu(x) over n values with the arithmetic of the GEMM's bias + GELU epilogues
// (bf16: the packed hardware-tanh form; fp32: gelu_f), so a recomputed activation
// equals, bit for bit, the one the forward pass fed to the next GEMM.
template <typename T> void gelu_recompute(T* y, const T* x, long long n, cudaStream_t s);
template <typename T> void to_storage(T* dst, const float* src, long long n, cudaStream_t s);
template <typename T> void to_f32(float* dst, const T* src, long long n, cudaStream_t s);

// Cross-entropy pieces.
template <typename T>
void ce_rowstats(const T* z, long long ldz, const int32_t* tgt, int M, int V, float* lse,
                 float* loss_rows, cudaStream_t s);
void ce_reduce_partials(const float* pmax, const float* psum, int ntiles, int ld, const float* ztgt,
                        int M, float* lse, float* loss_rows, cudaStream_t s);
template <typename T>
void ce_dlogits(T* z, long long ldz, const float* lse, const int32_t* tgt, int M, int V, int Vpad,
                float inv_scale, cudaStream_t s);
void mean_reduce(float* out, const float* rows, int M, unsigned* status, cudaStream_t s);

// Encoder backward: fixed-order scatter of dx0 (fp32) into dwte, and dwpe.
// dx0 is consumed: some of its rows are overwritten with partial sums.
void sort_tokens(uint32_t* order, const int32_t* tok, int M, int V, cudaStream_t s);
template <typename T>
void encoder_bwd(T* dwte, T* dwpe, float* dx0, const uint32_t* order, const int32_t* tok, int B,
                 int Tn, int C, cudaStream_t s);

// Split-K reduction: out = sum over splits of ws[s][m][n].
void splitk_reduce(void* out, int out_f32, long long ldo, const float* ws, int splits, int M, int N,
                   cudaStream_t s);

// Optimizer.
struct Segment { long long begin, end; int decay; };
constexpr int kMaxSegments = 16;
template <typename G>
void grad_sumsq_partials(float* partials, int nparts, const G* g, long long n, cudaStream_t s);
// Optimizer hyperparameters in device memory.  When the kernels below get a
// non-null `hp` they take lr, betas, eps, weight decay, max_norm and t from it
// instead of their value arguments (a captured CUDA graph then picks up new
// values from a host-to-device copy inside the graph).
struct OptHyper {
  float lr, b1, b2, eps, wd, max_norm;
  int t, pad;
};
// Update guard, device resident (llm.c GPT-2 1558M article: the long run skipped
// the parameter update when it saw a momentary spike, flags -sl / -sg; the run
// log prints a z-score beside the loss and the norm, "+nan" until it is defined).
// Each step's loss and gradient norm get a z-score against the previous `window`
// finite values of the same quantity (population mean and standard deviation;
// NaN while fewer than `window` values are held; 0 when the deviation is 0).
// The update is skipped when the loss or the norm is not finite, or when a
// threshold > 0 is set and that z-score exceeds it.
constexpr int kGuardMaxWindow = 256;
struct GuardState {
  float loss_z_max, norm_z_max;  // thresholds (<= 0: that check is off)
  int window;                    // values held for the statistics (2 .. kGuardMaxWindow)
  int count;                     // finite values held so far (<= window)
  int head;                      // next ring slot
  int skipped_spike;             // updates skipped for a z-score over its threshold
  int skipped_nonfinite;         // updates skipped for a non-finite loss or norm
  int last_skipped;              // 1 when the last update was skipped
  float z_loss, z_norm;          // z-scores of the last step
  float pad[6];
  float loss_hist[kGuardMaxWindow];
  float norm_hist[kGuardMaxWindow];
};
// norm_scale[0] = ||g||, [1] = clip scale, [2] = 1 - b1^t, [3] = 1 - b2^t, [4] = 1 when the
// update is skipped (then the step counter does not advance).  `loss`: the step's
// mean loss on the device; `guard` may be null (then only non-finite values skip).
void grad_norm_finalize(float* norm_scale, const float* partials, int nparts, float max_norm,
                        unsigned* status, int* counter, int host_t, float b1, float b2,
                        const OptHyper* hp, const float* loss, GuardState* guard, cudaStream_t s);
// bf16 mode: master/m/v fp32 with a bf16 copy of the parameters; fp32 mode: param_copy null.
template <typename G, typename P>
void adamw(float* master, P* param_copy, const G* grad, float* m, float* v, long long n,
           const Segment* segs, int nsegs, const float* norm_scale, float lr, float beta1,
           float beta2, float eps, float wd, const OptHyper* hp, cudaStream_t s);

}  // namespace gpt2k
