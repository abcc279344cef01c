// GPT-2 step sequencing and C ABI (see include/gpt2.h).
//
// The host code here carves one caller-owned device arena into parameters, AdamW
// state, every activation the backward pass needs and its scratch, then issues
// a fixed kernel sequence on the caller's stream.  Nothing is allocated after
// gpt2_create and no call synchronises unless a host output is requested, so
// the caller may capture forward + backward + clip_adamw in one CUDA graph.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "../../include/gpt2.h"

using namespace gpt2k;

namespace {
thread_local std::string g_last_cuda_error = "no error";
std::mutex g_once_mu;
int g_test_poison = 0;
}  // namespace

namespace gpt2k {

int test_poison() { return g_test_poison; }

int cuda_fail(cudaError_t e, const char* where) {
  g_last_cuda_error = std::string(where) + ": " + cudaGetErrorString(e);
  return GPT2_E_CUDA;
}

unsigned long long current_context_id() {
  typedef CUresult (*GetCurrent)(CUcontext*);
  typedef CUresult (*GetId)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag looked_up;
  std::call_once(looked_up, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (get_current(&c) != CUDA_SUCCESS || !c) return 0;
  if (get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

cudaError_t smem_limit_once(const void* kernel, int bytes, PerDeviceOnce* once) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_once_mu);
  const unsigned long long id = current_context_id();
  if (id != 0 && once->ctx[dev] == id) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  once->ctx[dev] = current_context_id();  // the call above made the context current if it was not
  return cudaSuccess;
}

}  // namespace gpt2k

namespace {
#define CK(call)                                        \
  do {                                                  \
    cudaError_t e_ = (call);                            \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
  } while (0)
#define CKI(call)                                                        \
  do {                                                                   \
    int e_ = (call);                                                     \
    if (e_ != 0) return cuda_fail((cudaError_t)e_, #call);               \
  } while (0)

struct Shape {
  int L, H, C, V, Vpad, T, B, prec;
  int rc = 0;  // activation recompute: 0 none, 1 GELU output, 2 GELU output and LayerNorm outputs
  int M() const { return B * T; }
  int d() const { return C / H; }
  size_t esz() const { return prec == GPT2_BF16 ? 2 : 4; }
};

// Canonical parameter tensors (names follow GPT-2); offsets in elements.
enum PIdx { P_WTE, P_WPE, P_LN1W, P_LN1B, P_QKVW, P_QKVB, P_APW, P_APB, P_LN2W, P_LN2B,
            P_FCW, P_FCB, P_FCPW, P_FCPB, P_LNFW, P_LNFB, P_COUNT };

struct ParamLayout {
  long long off[P_COUNT + 1];
  long long per_layer[P_COUNT];  // elements of one layer's slice (0 for non-layer tensors)
};

ParamLayout param_layout(int L, int C, int Vpad, int T) {
  long long sz[P_COUNT] = {
      (long long)Vpad * C, (long long)T * C, (long long)L * C, (long long)L * C,
      (long long)L * 3 * C * C, (long long)L * 3 * C, (long long)L * C * C, (long long)L * C,
      (long long)L * C, (long long)L * C, (long long)L * 4 * C * C, (long long)L * 4 * C,
      (long long)L * 4 * C * C, (long long)L * C, (long long)C, (long long)C};
  ParamLayout p;
  p.off[0] = 0;
  for (int i = 0; i < P_COUNT; ++i) p.off[i + 1] = p.off[i] + sz[i];
  for (int i = 0; i < P_COUNT; ++i) p.per_layer[i] = (i >= P_LN1W && i <= P_FCPB && L > 0) ? sz[i] / L : 0;
  return p;
}

bool is_decayed(int i) {
  return i == P_WTE || i == P_WPE || i == P_QKVW || i == P_APW || i == P_FCW || i == P_FCPW;
}

// Arena plan: byte offsets of every region, 256-byte aligned.
struct Plan {
  size_t total = 0;
  size_t params, grads, master, adam_m, adam_v, grad_acc;
  size_t tokens, targets;
  size_t res, x1, ln1, ln2, ln1_mean, ln1_rstd, ln2_mean, ln2_rstd, qkv, atty, att_lse, fch, fca;
  size_t lnf, lnf_mean, lnf_rstd, rc_stats, logits, ce_max, ce_sum, ce_tgt, ce_lse, ce_rows, scalars, status, hyper, guard;
  size_t dres, dres_b, dbig, dqkv, dsmall, attD, order, lnb_part, colsum_part, norm_part, sk_ws;
  size_t sk_bytes = 0;
  int ce_tiles = 0;
};

constexpr int kNormParts = 592;  // one wave of 512-thread blocks on 148 SMs (4 per SM)

size_t take(size_t& cur, size_t bytes) {
  size_t o = cur;
  cur += (bytes + 255) & ~size_t(255);
  return o;
}

Plan make_plan(const Shape& s) {
  Plan p;
  const size_t N = gpt2_num_params(s.L, s.C, s.Vpad, s.T);
  const size_t e = s.esz(), M = s.M(), C = s.C, L = s.L, f = 4;
  const bool bf = s.prec == GPT2_BF16;
  size_t cur = 0;
  p.params = take(cur, N * e);
  p.grads = take(cur, N * e);
  p.master = bf ? take(cur, N * f) : p.params;
  p.adam_m = take(cur, N * f);
  p.adam_v = take(cur, N * f);
  p.grad_acc = take(cur, N * f);
  p.tokens = take(cur, M * 4);
  p.targets = take(cur, M * 4);
  p.res = take(cur, (L + 1) * M * C * e);
  p.x1 = take(cur, L * M * C * e);
  // with LayerNorm recompute one buffer holds the LayerNorm output in use (forward: until
  // the next GEMM has read it; backward: recomputed for the weight-gradient GEMM)
  p.ln1 = take(cur, (s.rc >= 2 ? 1 : L) * M * C * e);
  p.ln2 = s.rc >= 2 ? p.ln1 : take(cur, L * M * C * e);
  p.ln1_mean = take(cur, L * M * f);
  p.ln1_rstd = take(cur, L * M * f);
  p.ln2_mean = take(cur, L * M * f);
  p.ln2_rstd = take(cur, L * M * f);
  p.qkv = take(cur, L * M * 3 * C * e);
  p.atty = take(cur, L * M * C * e);
  p.att_lse = take(cur, L * (size_t)s.B * s.H * s.T * f);
  p.fch = take(cur, L * M * 4 * C * e);
  // with GELU recompute one buffer holds gelu(h) in use (recomputed in the backward)
  p.fca = take(cur, (s.rc >= 1 ? 1 : L) * M * 4 * C * e);
  p.lnf = take(cur, M * C * e);
  p.lnf_mean = take(cur, M * f);
  p.lnf_rstd = take(cur, M * f);
  p.rc_stats = take(cur, 2 * M * f);  // statistics written by a recomputed LayerNorm (not read)
  p.logits = take(cur, M * (size_t)s.Vpad * e);
  p.ce_tiles = (s.Vpad + gemm_tc_stat_cols() - 1) / gemm_tc_stat_cols();
  p.ce_max = take(cur, M * p.ce_tiles * f);
  p.ce_sum = take(cur, M * p.ce_tiles * f);
  p.ce_tgt = take(cur, M * f);
  p.ce_lse = take(cur, M * f);
  p.ce_rows = take(cur, M * f);
  // [0] loss, [1] norm, [2] clip scale, [3..4] bias corrections, [5] update skipped,
  // [6] accumulated loss of gpt2_grad_accumulate, [8] step counter (int)
  p.scalars = take(cur, 16 * f);
  p.status = take(cur, 16);
  p.hyper = take(cur, sizeof(OptHyper));
  p.guard = take(cur, sizeof(GuardState));
  p.dres = take(cur, M * C * f);
  p.dres_b = bf ? take(cur, M * C * e) : p.dres;
  p.dbig = take(cur, M * 4 * C * e);
  p.dqkv = take(cur, M * 3 * C * e);
  p.dsmall = take(cur, M * C * e);
  p.attD = take(cur, (size_t)s.B * s.H * s.T * f);
  p.order = take(cur, 2 * M * 4);
  p.lnb_part = take(cur, layernorm_bwd_partials_floats(s.C) * f);
  // column-sum partials: the colsum kernel's, or the GELU' GEMM's one row per 32 rows
  size_t cs = std::max(colsum_partials_floats(4 * s.C), (size_t)((s.M() + 31) / 32) * 4 * s.C);
  cs = std::max(cs, (size_t)attn_bias_part_rows(s.B, s.T) * 3 * s.C);  // QKV bias partials of the attention backward
  p.colsum_part = take(cur, cs * f);
  p.norm_part = take(cur, kNormParts * f);
  // stream-K flags (zeroed with the arena) and partial-sum slots of the GEMM engine
  if (bf) p.sk_bytes = gemm_tc_sk_ws_bytes();
  p.sk_ws = take(cur, p.sk_bytes ? p.sk_bytes : 256);
  p.total = cur;
  return p;
}

int validate(const Shape& s) {
  if (s.L < 0 || s.H <= 0 || s.C <= 0 || s.V <= 0 || s.Vpad < s.V || s.T <= 0 || s.B <= 0)
    return GPT2_E_INVAL;
  if (s.prec != GPT2_FP32 && s.prec != GPT2_BF16) return GPT2_E_INVAL;
  if (s.C % s.H || s.C % 8 || s.Vpad % 8) return GPT2_E_INVAL;
  if ((long long)s.B * s.T > 16384) return GPT2_E_UNSUPPORTED;
  if (s.prec == GPT2_BF16 && (s.d() != 64 || s.C > 2048)) return GPT2_E_UNSUPPORTED;
  if (s.prec == GPT2_FP32 && (s.d() > 128 || s.C > 1024)) return GPT2_E_UNSUPPORTED;
  if (s.rc < 0 || s.rc > 2) return GPT2_E_INVAL;
  return GPT2_OK;
}

}  // namespace

struct ProfRec {
  int cls, ev0, ev1;
  double flops, bytes;
  int dims[6];  // GEMM regions: M, N, K, a_mn, b_mn, epilogue
};

struct gpt2 {
  Shape s;
  Plan p;
  ParamLayout pl;
  uint8_t* base;
  cudaStream_t stream;
  int state;  // 0 idle, 1 after forward, 2 after backward
  size_t N;
  // optional per-region CUDA-event timing (never while capturing a graph)
  bool prof_on = false;
  std::vector<cudaEvent_t> evpool;
  int evnext = 0;
  std::vector<ProfRec> recs;
  // gpt2_train_step_host: the whole step as one CUDA graph, captured on the first
  // call, fed from pinned staging buffers (tokens, targets, hyperparameters) and
  // writing loss, norm and status bits back to pinned memory
  cudaGraphExec_t host_exec = nullptr;
  cudaStream_t cap_stream = nullptr;
  int32_t* pin_tok = nullptr;
  int32_t* pin_tgt = nullptr;
  OptHyper* pin_hyp = nullptr;
  float* pin_out = nullptr;  // [0] loss, [1] norm, [2] status bits
  // update guard settings (thresholds <= 0: off; the device state lives in the arena)
  float guard_loss_z = 0.f, guard_norm_z = 0.f;
  int guard_window = 0;
  template <typename T> T* at(size_t off) const { return reinterpret_cast<T*>(base + off); }
};

// acc = (first ? 0 : acc) + scale * g over n values (fp32 accumulator; mem_kernels.cu).
namespace gpt2k {
template <typename G>
void grad_accumulate(float* acc, const G* g, long long n, float scale, int first, const float* loss,
                     float* acc_loss, cudaStream_t s);
}  // namespace gpt2k

namespace {

enum { ST_IDLE = 0, ST_FWD = 1, ST_BWD = 2, ST_ACC = 3 };

int prof_begin(gpt2* h) {
  if (!h->prof_on || h->evnext + 2 > (int)h->evpool.size()) return -1;
  cudaEventRecord(h->evpool[h->evnext], h->stream);
  return h->evnext++;
}
void prof_end(gpt2* h, int i0, int cls, double flops, double bytes, const int* dims = nullptr) {
  if (i0 < 0) return;
  cudaEventRecord(h->evpool[h->evnext], h->stream);
  ProfRec r{cls, i0, h->evnext, flops, bytes, {0, 0, 0, 0, 0, 0}};
  if (dims)
    for (int i = 0; i < 6; ++i) r.dims[i] = dims[i];
  h->recs.push_back(r);
  h->evnext++;
}
// Run `stmt` as one timed region of kernel class `cls` with its algorithmic flops / bytes.
#define REGION(cls, flops, bytes, ...)           \
  do {                                           \
    int pi_ = prof_begin(h);                     \
    __VA_ARGS__;                                 \
    prof_end(h, pi_, (cls), (flops), (bytes));   \
  } while (0)

template <typename T>
struct Ptrs {
  const gpt2* h;
  explicit Ptrs(const gpt2* hh) : h(hh) {}
  T* param(int i, int l = 0) const {
    return h->at<T>(h->p.params) + h->pl.off[i] + (long long)l * h->pl.per_layer[i];
  }
  T* grad(int i, int l = 0) const {
    return h->at<T>(h->p.grads) + h->pl.off[i] + (long long)l * h->pl.per_layer[i];
  }
  long long MC() const { return (long long)h->s.M() * h->s.C; }
  T* res(int l) const { return h->at<T>(h->p.res) + l * MC(); }
  T* x1(int l) const { return h->at<T>(h->p.x1) + l * MC(); }
  T* ln1(int l) const { return h->at<T>(h->p.ln1) + (h->s.rc >= 2 ? 0 : l) * MC(); }
  T* ln2(int l) const { return h->at<T>(h->p.ln2) + (h->s.rc >= 2 ? 0 : l) * MC(); }
  T* qkv(int l) const { return h->at<T>(h->p.qkv) + l * 3 * MC(); }
  T* atty(int l) const { return h->at<T>(h->p.atty) + l * MC(); }
  T* fch(int l) const { return h->at<T>(h->p.fch) + l * 4 * MC(); }
  T* fca(int l) const { return h->at<T>(h->p.fca) + (h->s.rc >= 1 ? 0 : l) * 4 * MC(); }
  float* stat(size_t region, int l) const { return h->at<float>(region) + (long long)l * h->s.M(); }
  float* att_lse(int l) const {
    return h->at<float>(h->p.att_lse) + (long long)l * h->s.B * h->s.H * h->s.T;
  }
};

// One Linear through the precision's GEMM engine (bf16: stream-K schedule where it pays).
template <typename T>
int linear(gpt2* h, GemmArgs g) {
  unsigned* status = h->at<unsigned>(h->p.status);
  const double flops = 2.0 * g.M * g.N * (double)g.K;
  const double bytes = ((double)g.M * g.K + (double)g.N * g.K + (double)g.M * g.N) * sizeof(T);
  int e = 0;
  const int dims[6] = {g.M, g.N, g.K, g.a_mn, g.b_mn, g.epi};
  if (sizeof(T) == 2) {
    int rs = 0;
    const int pi = prof_begin(h);
    e = gemm_tc(g, GEMM_TC_STREAM_K, h->at<void>(h->p.sk_ws), h->p.sk_bytes, status, h->stream, 0, &rs);
    prof_end(h, pi, GPT2_K_GEMM, flops, bytes, dims);
    if (e) return e;
    if (rs > 1)
      REGION(GPT2_K_SPLITK, 0.0, (double)g.M * g.N * (4.0 * rs + 2.0),
             splitk_reduce(g.D, g.epi == EPI_F32, g.ldd,
                           reinterpret_cast<float*>(h->at<char>(h->p.sk_ws) + gemm_tc_sk_plane_offset()), rs,
                           g.M, g.N, h->stream));
    return (int)cudaGetLastError();
  }
  const int pi = prof_begin(h);
  e = gemm_simt(g, h->stream);
  prof_end(h, pi, GPT2_K_GEMM, flops, bytes, dims);
  return e;
}

template <typename T>
int forward_impl(gpt2* h) {
  const Shape& s = h->s;
  Ptrs<T> P(h);
  const int M = s.M(), C = s.C, L = s.L;
  const double E = sizeof(T), MC = (double)M * C;
  cudaStream_t st = h->stream;
  unsigned* status = h->at<unsigned>(h->p.status);
  int32_t* tok = h->at<int32_t>(h->p.tokens);
  int32_t* tgt = h->at<int32_t>(h->p.targets);
  const double attn_flops = 4.0 * s.B * s.H * (double)s.d() * s.T * (s.T + 1) / 2.0;
  REGION(GPT2_K_ENCODER, 0.0, 2.0 * MC * E + 2.0 * MC * E + 8.0 * M, {
    check_ids(tok, M, s.V, status, st);
    check_ids(tgt, M, s.V, status, st);
    encoder_fwd<T>(P.res(0), tok, P.param(P_WTE), P.param(P_WPE), s.B, s.T, C, s.V, status, st);
  });
  for (int l = 0; l < L; ++l) {
    T* x = P.res(l);
    REGION(GPT2_K_LN_FWD, 0.0, 2.0 * MC * E + 8.0 * M,
           layernorm_fwd<T>(P.ln1(l), P.stat(h->p.ln1_mean, l), P.stat(h->p.ln1_rstd, l), x,
                            P.param(P_LN1W, l), P.param(P_LN1B, l), M, C, st));
    GemmArgs g;
    g.A = P.ln1(l); g.lda = C; g.B = P.param(P_QKVW, l); g.ldb = C;
    g.M = M; g.N = 3 * C; g.K = C; g.epi = EPI_BIAS; g.D = P.qkv(l); g.ldd = 3 * C;
    g.bias = P.param(P_QKVB, l);
    CKI(linear<T>(h, g));
    AttnArgs a;
    T* qkv = P.qkv(l);
    a.q = qkv; a.k = qkv + C; a.v = qkv + 2 * C; a.o = P.atty(l); a.lse = P.att_lse(l);
    a.B = s.B; a.H = s.H; a.T = s.T; a.d = s.d();
    a.sb = (long long)s.T * 3 * C; a.sh = s.d(); a.st = 3 * C;
    a.osb = (long long)s.T * C; a.osh = s.d(); a.ost = C;
    a.scale = 1.0f / sqrtf((float)s.d());
    a.status = status;
    int e = 0;
    REGION(GPT2_K_ATTN_FWD, attn_flops, 4.0 * MC * E,
           e = (sizeof(T) == 2 ? attn_fwd_tc(a, st) : attn_fwd_f32(a, st)));
    CKI(e);
    g = GemmArgs();
    g.A = P.atty(l); g.lda = C; g.B = P.param(P_APW, l); g.ldb = C;
    g.M = M; g.N = C; g.K = C; g.epi = EPI_BIAS_RESID; g.D = P.x1(l); g.ldd = C;
    g.bias = P.param(P_APB, l); g.resid = x; g.ldr = C;
    CKI(linear<T>(h, g));
    REGION(GPT2_K_LN_FWD, 0.0, 2.0 * MC * E + 8.0 * M,
           layernorm_fwd<T>(P.ln2(l), P.stat(h->p.ln2_mean, l), P.stat(h->p.ln2_rstd, l), P.x1(l),
                            P.param(P_LN2W, l), P.param(P_LN2B, l), M, C, st));
    g = GemmArgs();
    g.A = P.ln2(l); g.lda = C; g.B = P.param(P_FCW, l); g.ldb = C;
    // fch keeps gelu'(h) for the backward, or h itself when the backward recomputes
    g.M = M; g.N = 4 * C; g.K = C; g.epi = s.rc >= 1 ? EPI_BIAS_GELU_H : EPI_BIAS_GELU; g.D = P.fch(l);
    g.ldd = 4 * C; g.D2 = P.fca(l); g.bias = P.param(P_FCB, l);
    CKI(linear<T>(h, g));
    g = GemmArgs();
    g.A = P.fca(l); g.lda = 4 * C; g.B = P.param(P_FCPW, l); g.ldb = 4 * C;
    g.M = M; g.N = C; g.K = 4 * C; g.epi = EPI_BIAS_RESID; g.D = P.res(l + 1); g.ldd = C;
    g.bias = P.param(P_FCPB, l); g.resid = P.x1(l); g.ldr = C;
    CKI(linear<T>(h, g));
  }
  T* lnf = h->at<T>(h->p.lnf);
  REGION(GPT2_K_LN_FWD, 0.0, 2.0 * MC * E + 8.0 * M,
         layernorm_fwd<T>(lnf, h->at<float>(h->p.lnf_mean), h->at<float>(h->p.lnf_rstd), P.res(L),
                          P.param(P_LNFW), P.param(P_LNFB), M, C, st));
  // tied lm_head + cross-entropy; the logits become dlogits in place
  T* logits = h->at<T>(h->p.logits);
  float* lse = h->at<float>(h->p.ce_lse);
  float* rows = h->at<float>(h->p.ce_rows);
  const double zbytes = (double)M * s.Vpad * E;
  GemmArgs g;
  g.A = lnf; g.lda = C; g.B = P.param(P_WTE); g.ldb = C;
  g.M = M; g.N = s.Vpad; g.K = C; g.D = logits; g.ldd = s.Vpad;
  if (sizeof(T) == 2) {
    g.epi = EPI_CE;
    g.ce_max = h->at<float>(h->p.ce_max); g.ce_sum = h->at<float>(h->p.ce_sum);
    g.ce_ld = h->p.ce_tiles; g.ce_tgt = h->at<float>(h->p.ce_tgt); g.targets = tgt; g.V = s.V;
    CKI(linear<T>(h, g));
    REGION(GPT2_K_CE, 0.0, 8.0 * M * h->p.ce_tiles + 16.0 * M,
           ce_reduce_partials(g.ce_max, g.ce_sum, h->p.ce_tiles, h->p.ce_tiles, g.ce_tgt, M, lse, rows, st));
  } else {
    g.epi = EPI_STORE;
    CKI(linear<T>(h, g));
    REGION(GPT2_K_CE, 0.0, zbytes, ce_rowstats<T>(logits, s.Vpad, tgt, M, s.V, lse, rows, st));
  }
  REGION(GPT2_K_CE, 0.0, 2.0 * zbytes + 12.0 * M, {
    mean_reduce(h->at<float>(h->p.scalars), rows, M, status, st);
    ce_dlogits<T>(logits, s.Vpad, lse, tgt, M, s.V, s.Vpad, 1.0f / (float)M, st);
  });
  CK(cudaGetLastError());
  return GPT2_OK;
}

template <typename T>
int backward_impl(gpt2* h) {
  const Shape& s = h->s;
  Ptrs<T> P(h);
  const int M = s.M(), C = s.C, L = s.L;
  const double E = sizeof(T), MC = (double)M * C;
  cudaStream_t st = h->stream;
  const bool bf = sizeof(T) == 2;
  T* dz = h->at<T>(h->p.logits);
  T* lnf = h->at<T>(h->p.lnf);
  T* dsmall = h->at<T>(h->p.dsmall);
  T* dbig = h->at<T>(h->p.dbig);
  T* dqkv = h->at<T>(h->p.dqkv);
  float* dres = h->at<float>(h->p.dres);
  T* dres_b = bf ? h->at<T>(h->p.dres_b) : nullptr;
  T* dcur = bf ? dres_b : reinterpret_cast<T*>(dres);
  float* lnbp = h->at<float>(h->p.lnb_part);
  float* csp = h->at<float>(h->p.colsum_part);
  const double attn_flops = 2.5 * 4.0 * s.B * s.H * (double)s.d() * s.T * (s.T + 1) / 2.0;
  // LN backward bytes: dy, x (storage), dres read+write fp32, dres copy, mean/rstd
  const double lnb_first = 2.0 * MC * E + 4.0 * MC + (bf ? MC * E : 0.0) + 8.0 * M;
  const double lnb_acc = lnb_first + 4.0 * MC;
  // classifier: dlnf = dz wte ; dwte = dz^T lnf
  GemmArgs g;
  g.A = dz; g.lda = s.Vpad; g.B = P.param(P_WTE); g.ldb = C; g.b_mn = 1;
  g.M = M; g.N = C; g.K = s.Vpad; g.D = dsmall; g.ldd = C;
  CKI(linear<T>(h, g));
  g = GemmArgs();
  g.A = dz; g.lda = s.Vpad; g.a_mn = 1; g.B = lnf; g.ldb = C; g.b_mn = 1;
  g.M = s.Vpad; g.N = C; g.K = M; g.D = P.grad(P_WTE); g.ldd = C;
  CKI(linear<T>(h, g));
  REGION(GPT2_K_LN_BWD, 0.0, lnb_first,
         layernorm_bwd<T>(dres, dres_b, dsmall, P.res(L), h->at<float>(h->p.lnf_mean),
                          h->at<float>(h->p.lnf_rstd), P.param(P_LNFW), P.grad(P_LNFW),
                          P.grad(P_LNFB), L > 0 ? P.grad(P_FCPB, L - 1) : nullptr, lnbp, M, C, 0,
                          st, h->at<unsigned>(h->p.status)));
  for (int l = L - 1; l >= 0; --l) {
    if (s.rc >= 1)  // gelu(h) for the projection's weight gradient, from the h the forward kept
      REGION(GPT2_K_RECOMPUTE, 0.0, 2.0 * 4.0 * MC * E, gelu_recompute<T>(P.fca(l), P.fch(l), (long long)4 * M * C, st));
    // MLP projection: x2 = x1 + fca Wfcp^T + b
    g = GemmArgs();
    g.A = dcur; g.lda = C; g.a_mn = 1; g.B = P.fca(l); g.ldb = 4 * C; g.b_mn = 1;
    g.M = C; g.N = 4 * C; g.K = M; g.D = P.grad(P_FCPW, l); g.ldd = 4 * C;
    CKI(linear<T>(h, g));
    // the fcproj bias gradient (column sum of dcur) came out of the previous LayerNorm backward
    g = GemmArgs();
    g.A = dcur; g.lda = C; g.B = P.param(P_FCPW, l); g.ldb = 4 * C; g.b_mn = 1;
    g.M = M; g.N = 4 * C; g.K = C; g.epi = s.rc >= 1 ? EPI_GELU_BWD_H : EPI_GELU_BWD; g.aux = P.fch(l);
    g.ldaux = 4 * C;
    g.D = dbig; g.ldd = 4 * C;
    if (bf) g.colpart = csp;  // the fc bias gradient's partial column sums come out of this epilogue
    CKI(linear<T>(h, g));
    // MLP up-projection: h = ln2 Wfc^T + b
    if (s.rc >= 2)
      REGION(GPT2_K_RECOMPUTE, 0.0, 2.0 * MC * E + 8.0 * M,
             layernorm_fwd<T>(P.ln2(l), h->at<float>(h->p.rc_stats), h->at<float>(h->p.rc_stats) + M, P.x1(l),
                              P.param(P_LN2W, l), P.param(P_LN2B, l), M, C, st));
    g = GemmArgs();
    g.A = dbig; g.lda = 4 * C; g.a_mn = 1; g.B = P.ln2(l); g.ldb = C; g.b_mn = 1;
    g.M = 4 * C; g.N = C; g.K = M; g.D = P.grad(P_FCW, l); g.ldd = C;
    CKI(linear<T>(h, g));
    if (bf)
      REGION(GPT2_K_BIAS_GRAD, 0.0, 4.0 * ((M + 31) / 32) * 4.0 * C,
             colsum_reduce<T>(P.grad(P_FCB, l), csp, (M + 31) / 32, 4 * C, st));
    else
      REGION(GPT2_K_BIAS_GRAD, 0.0, 4.0 * MC * E, colsum<T>(P.grad(P_FCB, l), dbig, M, 4 * C, 4 * C, csp, st));
    g = GemmArgs();
    g.A = dbig; g.lda = 4 * C; g.B = P.param(P_FCW, l); g.ldb = C; g.b_mn = 1;
    g.M = M; g.N = C; g.K = 4 * C; g.D = dsmall; g.ldd = C;
    CKI(linear<T>(h, g));
    REGION(GPT2_K_LN_BWD, 0.0, lnb_acc,
           layernorm_bwd<T>(dres, dres_b, dsmall, P.x1(l), P.stat(h->p.ln2_mean, l),
                            P.stat(h->p.ln2_rstd, l), P.param(P_LN2W, l), P.grad(P_LN2W, l),
                            P.grad(P_LN2B, l), P.grad(P_APB, l), lnbp, M, C, 1, st, h->at<unsigned>(h->p.status)));
    // attention projection: x1 = x + atty Wap^T + b
    g = GemmArgs();
    g.A = dcur; g.lda = C; g.a_mn = 1; g.B = P.atty(l); g.ldb = C; g.b_mn = 1;
    g.M = C; g.N = C; g.K = M; g.D = P.grad(P_APW, l); g.ldd = C;
    CKI(linear<T>(h, g));
    g = GemmArgs();
    g.A = dcur; g.lda = C; g.B = P.param(P_APW, l); g.ldb = C; g.b_mn = 1;
    g.M = M; g.N = C; g.K = C; g.D = dsmall; g.ldd = C;
    CKI(linear<T>(h, g));
    // attention
    AttnArgs a;
    T* qkv = P.qkv(l);
    a.q = qkv; a.k = qkv + C; a.v = qkv + 2 * C; a.o = P.atty(l); a.lse = P.att_lse(l);
    a.dO = dsmall; a.dq = dqkv; a.dk = dqkv + C; a.dv = dqkv + 2 * C;
    a.Dbuf = h->at<float>(h->p.attD);
    a.B = s.B; a.H = s.H; a.T = s.T; a.d = s.d();
    a.sb = (long long)s.T * 3 * C; a.sh = s.d(); a.st = 3 * C;
    a.osb = (long long)s.T * C; a.osh = s.d(); a.ost = C;
    a.scale = 1.0f / sqrtf((float)s.d());
    a.status = h->at<unsigned>(h->p.status);
    if (bf) a.bias_part = csp;  // the QKV bias gradient's partial column sums
    int e = 0;
    REGION(GPT2_K_ATTN_BWD, attn_flops, 8.0 * MC * E, e = (bf ? attn_bwd_bf16(a, st) : attn_bwd_f32(a, st)));
    CKI(e);
    // QKV: qkv = ln1 Wqkv^T + b
    if (s.rc >= 2)
      REGION(GPT2_K_RECOMPUTE, 0.0, 2.0 * MC * E + 8.0 * M,
             layernorm_fwd<T>(P.ln1(l), h->at<float>(h->p.rc_stats), h->at<float>(h->p.rc_stats) + M, P.res(l),
                              P.param(P_LN1W, l), P.param(P_LN1B, l), M, C, st));
    g = GemmArgs();
    g.A = dqkv; g.lda = 3 * C; g.a_mn = 1; g.B = P.ln1(l); g.ldb = C; g.b_mn = 1;
    g.M = 3 * C; g.N = C; g.K = M; g.D = P.grad(P_QKVW, l); g.ldd = C;
    CKI(linear<T>(h, g));
    if (bf)
      REGION(GPT2_K_BIAS_GRAD, 0.0, 4.0 * attn_bias_part_rows(s.B, s.T) * 3.0 * C,
             colsum_reduce<T>(P.grad(P_QKVB, l), csp, attn_bias_part_rows(s.B, s.T), 3 * C, st));
    else
      REGION(GPT2_K_BIAS_GRAD, 0.0, 3.0 * MC * E, colsum<T>(P.grad(P_QKVB, l), dqkv, M, 3 * C, 3 * C, csp, st));
    g = GemmArgs();
    g.A = dqkv; g.lda = 3 * C; g.B = P.param(P_QKVW, l); g.ldb = C; g.b_mn = 1;
    g.M = M; g.N = C; g.K = 3 * C; g.D = dsmall; g.ldd = C;
    CKI(linear<T>(h, g));
    REGION(GPT2_K_LN_BWD, 0.0, lnb_acc,
           layernorm_bwd<T>(dres, dres_b, dsmall, P.res(l), P.stat(h->p.ln1_mean, l),
                            P.stat(h->p.ln1_rstd, l), P.param(P_LN1W, l), P.grad(P_LN1W, l),
                            P.grad(P_LN1B, l), l > 0 ? P.grad(P_FCPB, l - 1) : nullptr, lnbp, M, C,
                            1, st, h->at<unsigned>(h->p.status)));
  }
  // encoder: dwte[tok] += dx0 in a fixed order, dwpe = sum over the batch
  uint32_t* order = h->at<uint32_t>(h->p.order);
  REGION(GPT2_K_ENCODER, 0.0, 4.0 * MC + 2.0 * (double)s.T * C * E, {
    sort_tokens(order, h->at<int32_t>(h->p.tokens), M, s.V, st);
    encoder_bwd<T>(P.grad(P_WTE), P.grad(P_WPE), dres, order, h->at<int32_t>(h->p.tokens), s.B,
                   s.T, C, st);
  });
  CK(cudaGetLastError());
  return GPT2_OK;
}

// Clip + AdamW with gradients g of type G: the step's storage-type gradients, or
// the fp32 accumulator of gpt2_grad_accumulate.
template <typename T, typename G>
int clip_adamw_grads(gpt2* h, const G* g, const float* loss, float lr, float b1, float b2, float eps, float wd,
                     float max_norm, int t, const OptHyper* hp) {
  cudaStream_t st = h->stream;
  float* ns = h->at<float>(h->p.scalars) + 1;
  int* counter = reinterpret_cast<int*>(h->at<float>(h->p.scalars) + 8);
  float* np_ = h->at<float>(h->p.norm_part);
  unsigned* status = h->at<unsigned>(h->p.status);
  const double N = (double)h->N, E = sizeof(T), EG = sizeof(G);
  REGION(GPT2_K_NORM, 0.0, N * EG, {
    grad_sumsq_partials<G>(np_, kNormParts, g, (long long)h->N, st);
    grad_norm_finalize(ns, np_, kNormParts, max_norm, status, counter, t, b1, b2, hp, loss,
                       h->at<GuardState>(h->p.guard), st);
  });
  Segment segs[P_COUNT];
  for (int i = 0; i < P_COUNT; ++i) segs[i] = Segment{h->pl.off[i], h->pl.off[i + 1], is_decayed(i) ? 1 : 0};
  T* pcopy = sizeof(T) == 2 ? h->at<T>(h->p.params) : nullptr;
  // master, m, v read + written (fp32), gradient read, bf16 copy written
  const double bytes = N * (24.0 + EG + (sizeof(T) == 2 ? E : 0.0));
  REGION(GPT2_K_ADAMW, 0.0, bytes,
         adamw<G, T>(h->at<float>(h->p.master), pcopy, g, h->at<float>(h->p.adam_m), h->at<float>(h->p.adam_v),
                     (long long)h->N, segs, P_COUNT, ns, lr, b1, b2, eps, wd, hp, st));
  CK(cudaGetLastError());
  return GPT2_OK;
}

template <typename T>
int clip_adamw_impl(gpt2* h, float lr, float b1, float b2, float eps, float wd, float max_norm,
                    int t, const OptHyper* hp = nullptr) {
  return clip_adamw_grads<T, T>(h, h->at<T>(h->p.grads), h->at<float>(h->p.scalars), lr, b1, b2, eps, wd,
                                max_norm, t, hp);
}

// After an expired bounded wait a GEMM may have left stream-K flags raised;
// lower them all so the next launch starts from a clean workspace.
int clear_sk_flags(gpt2* h) {
  if (h->p.sk_bytes) CK(cudaMemsetAsync(h->at<char>(h->p.sk_ws), 0, gemm_tc_sk_plane_offset(), h->stream));
  return GPT2_OK;
}

constexpr int kGuardDefaultWindow = 128;

// Uploads a fresh update-guard state (empty window, zero counters) with these settings.
int reset_guard(gpt2* h, float loss_z, float norm_z, int window) {
  GuardState g;
  memset(&g, 0, sizeof(g));
  g.loss_z_max = loss_z;
  g.norm_z_max = norm_z;
  g.window = window;
  const float nan = __builtin_nanf("");
  g.z_loss = nan;
  g.z_norm = nan;
  h->guard_loss_z = loss_z;
  h->guard_norm_z = norm_z;
  h->guard_window = window;
  CK(cudaMemcpyAsync(h->at<GuardState>(h->p.guard), &g, sizeof(g), cudaMemcpyHostToDevice, h->stream));
  // the source is a stack object: finish the copy before it goes out of scope
  CK(cudaStreamSynchronize(h->stream));
  return GPT2_OK;
}

int read_status(gpt2* h) {
  unsigned st = 0;
  CK(cudaStreamSynchronize(h->stream));
  CK(cudaMemcpy(&st, h->at<unsigned>(h->p.status), 4, cudaMemcpyDeviceToHost));
  if (st) CK(cudaMemsetAsync(h->at<unsigned>(h->p.status), 0, 4, h->stream));
  if (st & ST_TIMEOUT) {
    clear_sk_flags(h);
    return GPT2_E_TIMEOUT;
  }
  if (st & ST_TOKEN) return GPT2_E_TOKEN;
  if (st & ST_NONFINITE) return GPT2_E_NONFINITE;
  return GPT2_OK;
}

}  // namespace

// ====================================================================== C ABI
extern "C" {

size_t gpt2_num_params(int L, int C, int Vpad, int T) {
  if (L < 0 || C <= 0 || Vpad <= 0 || T <= 0) return 0;
  return (size_t)Vpad * C + (size_t)T * C + (size_t)L * (12 * (size_t)C * C + 13 * (size_t)C) + 2 * (size_t)C;
}

size_t gpt2_arena_bytes_r(int L, int H, int C, int V, int Vpad, int T, int B, int precision, int recompute) {
  Shape s{L, H, C, V, Vpad, T, B, precision, recompute};
  if (validate(s) != GPT2_OK) return 0;
  return make_plan(s).total;
}

size_t gpt2_arena_bytes(int L, int H, int C, int V, int Vpad, int T, int B, int precision) {
  return gpt2_arena_bytes_r(L, H, C, V, Vpad, T, B, precision, 0);
}

int gpt2_create(int L, int H, int C, int V, int Vpad, int T, int B, int precision, void* d_arena,
                size_t arena_bytes, void* stream, gpt2_t** out) {
  return gpt2_create_r(L, H, C, V, Vpad, T, B, precision, 0, d_arena, arena_bytes, stream, out);
}

int gpt2_create_r(int L, int H, int C, int V, int Vpad, int T, int B, int precision, int recompute, void* d_arena,
                  size_t arena_bytes, void* stream, gpt2_t** out) {
  if (!out) return GPT2_E_INVAL;
  *out = nullptr;
  Shape s{L, H, C, V, Vpad, T, B, precision, recompute};
  int v = validate(s);
  if (v != GPT2_OK) return v;
  if (!d_arena || (reinterpret_cast<uintptr_t>(d_arena) & 255)) return GPT2_E_INVAL;
  Plan p = make_plan(s);
  if (arena_bytes < p.total) return GPT2_E_INVAL;
  gpt2* h = new gpt2();
  h->s = s;
  h->p = p;
  h->pl = param_layout(L, C, Vpad, T);
  h->base = static_cast<uint8_t*>(d_arena);
  h->stream = static_cast<cudaStream_t>(stream);
  h->state = ST_IDLE;
  h->N = gpt2_num_params(L, C, Vpad, T);
  cudaError_t e = cudaMemsetAsync(d_arena, 0, p.total, h->stream);
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e, "gpt2_create memset");
  }
  int r = reset_guard(h, 0.f, 0.f, kGuardDefaultWindow);
  if (r != GPT2_OK) {
    delete h;
    return r;
  }
  *out = h;
  return GPT2_OK;
}

void gpt2_destroy(gpt2_t* h) {
  if (!h) return;
  for (cudaEvent_t e : h->evpool) cudaEventDestroy(e);
  if (h->host_exec) cudaGraphExecDestroy(h->host_exec);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  if (h->pin_tok) cudaFreeHost(h->pin_tok);
  if (h->pin_tgt) cudaFreeHost(h->pin_tgt);
  if (h->pin_hyp) cudaFreeHost(h->pin_hyp);
  if (h->pin_out) cudaFreeHost(h->pin_out);
  delete h;
}

int gpt2_profile(gpt2_t* h, int on) {
  if (!h) return GPT2_E_INVAL;
  if (on) {
    if (h->evpool.empty()) {
      h->evpool.resize(65536);  // two events per region: enough for several steps of the 48-layer model
      for (auto& e : h->evpool) CK(cudaEventCreate(&e));
    }
    h->recs.clear();
    h->evnext = 0;
  }
  h->prof_on = on != 0;
  return GPT2_OK;
}

int gpt2_profile_regions(gpt2_t* h) {
  if (!h) return GPT2_E_INVAL;
  return (int)h->recs.size();
}

int gpt2_profile_region(gpt2_t* h, int i, int* kernel_class, int* dims, double* ms, double* flops,
                        double* bytes) {
  if (!h || i < 0 || i >= (int)h->recs.size()) return GPT2_E_INVAL;
  CK(cudaStreamSynchronize(h->stream));
  const ProfRec& r = h->recs[i];
  float x = 0.f;
  CK(cudaEventElapsedTime(&x, h->evpool[r.ev0], h->evpool[r.ev1]));
  if (kernel_class) *kernel_class = r.cls;
  if (dims)
    for (int k = 0; k < 6; ++k) dims[k] = r.dims[k];
  if (ms) *ms = x;
  if (flops) *flops = r.flops;
  if (bytes) *bytes = r.bytes;
  return GPT2_OK;
}

int gpt2_profile_read(gpt2_t* h, int kernel_class, int* regions, double* ms, double* flops,
                      double* bytes) {
  if (!h || kernel_class < 0 || kernel_class >= GPT2_K_COUNT) return GPT2_E_INVAL;
  CK(cudaStreamSynchronize(h->stream));
  int n = 0;
  double t = 0, f = 0, b = 0;
  for (const ProfRec& r : h->recs) {
    if (r.cls != kernel_class) continue;
    float x = 0.f;
    CK(cudaEventElapsedTime(&x, h->evpool[r.ev0], h->evpool[r.ev1]));
    ++n;
    t += x;
    f += r.flops;
    b += r.bytes;
  }
  if (regions) *regions = n;
  if (ms) *ms = t;
  if (flops) *flops = f;
  if (bytes) *bytes = b;
  return GPT2_OK;
}

int gpt2_set_stream(gpt2_t* h, void* stream) {
  if (!h) return GPT2_E_INVAL;
  h->stream = static_cast<cudaStream_t>(stream);
  return GPT2_OK;
}

int gpt2_set_params(gpt2_t* h, const float* params, int on_device) {
  if (!h || !params) return GPT2_E_INVAL;
  const size_t bytes = h->N * 4;
  float* master = h->at<float>(h->p.master);
  CK(cudaMemcpyAsync(master, params, bytes, on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice,
                     h->stream));
  if (h->s.prec == GPT2_BF16) to_storage<bf16>(h->at<bf16>(h->p.params), master, (long long)h->N, h->stream);
  CK(cudaMemsetAsync(h->at<float>(h->p.adam_m), 0, bytes, h->stream));
  CK(cudaMemsetAsync(h->at<float>(h->p.adam_v), 0, bytes, h->stream));
  CK(cudaMemsetAsync(h->at<float>(h->p.scalars), 0, 16 * sizeof(float), h->stream));  // step counter
  CK(cudaGetLastError());
  if (!on_device) CK(cudaStreamSynchronize(h->stream));
  h->state = ST_IDLE;
  return GPT2_OK;
}

int gpt2_get_tensor(gpt2_t* h, int which, float* dst, int dst_on_device) {
  if (!h || !dst) return GPT2_E_INVAL;
  const bool bf = h->s.prec == GPT2_BF16;
  size_t off;
  bool storage = false;
  switch (which) {
    case GPT2_PARAMS: off = h->p.params; storage = bf; break;
    case GPT2_GRADS: off = h->p.grads; storage = bf; break;
    case GPT2_ADAM_M: off = h->p.adam_m; break;
    case GPT2_ADAM_V: off = h->p.adam_v; break;
    case GPT2_MASTER: off = h->p.master; break;
    case GPT2_GRAD_ACC: off = h->p.grad_acc; break;
    default: return GPT2_E_INVAL;
  }
  const size_t n = h->N;
  if (!storage) {
    CK(cudaMemcpyAsync(dst, h->at<float>(off), n * 4,
                       dst_on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyDeviceToHost, h->stream));
    if (!dst_on_device) CK(cudaStreamSynchronize(h->stream));
    return GPT2_OK;
  }
  if (dst_on_device) {
    to_f32<bf16>(dst, h->at<bf16>(off), (long long)n, h->stream);
    CK(cudaGetLastError());
    return GPT2_OK;
  }
  std::vector<uint16_t> tmp(n);
  CK(cudaMemcpyAsync(tmp.data(), h->at<void>(off), n * 2, cudaMemcpyDeviceToHost, h->stream));
  CK(cudaStreamSynchronize(h->stream));
  for (size_t i = 0; i < n; ++i) {
    uint32_t u = (uint32_t)tmp[i] << 16;
    memcpy(dst + i, &u, 4);
  }
  return GPT2_OK;
}

int gpt2_forward(gpt2_t* h, const int32_t* d_tokens, const int32_t* d_targets, float* h_loss) {
  if (!h || !d_tokens || !d_targets) return GPT2_E_INVAL;
  const size_t bytes = (size_t)h->s.M() * 4;
  CK(cudaMemcpyAsync(h->at<int32_t>(h->p.tokens), d_tokens, bytes, cudaMemcpyDeviceToDevice, h->stream));
  CK(cudaMemcpyAsync(h->at<int32_t>(h->p.targets), d_targets, bytes, cudaMemcpyDeviceToDevice, h->stream));
  int r = h->s.prec == GPT2_BF16 ? forward_impl<bf16>(h) : forward_impl<float>(h);
  if (r != GPT2_OK) return r;
  h->state = ST_FWD;
  if (h_loss) {
    int st = read_status(h);
    CK(cudaMemcpy(h_loss, h->at<float>(h->p.scalars), 4, cudaMemcpyDeviceToHost));
    if (st != GPT2_OK) return st;
  }
  return GPT2_OK;
}

int gpt2_backward(gpt2_t* h) {
  if (!h) return GPT2_E_INVAL;
  if (h->state != ST_FWD) return GPT2_E_STATE;
  int r = h->s.prec == GPT2_BF16 ? backward_impl<bf16>(h) : backward_impl<float>(h);
  if (r != GPT2_OK) return r;
  h->state = ST_BWD;
  return GPT2_OK;
}

int gpt2_clip_adamw(gpt2_t* h, float lr, float beta1, float beta2, float eps, float weight_decay,
                    float max_norm, int step_t, float* h_norm) {
  if (!h) return GPT2_E_INVAL;
  if (step_t < 0 || !(max_norm > 0.f)) return GPT2_E_INVAL;
  if (h->state != ST_BWD) return GPT2_E_STATE;
  int r = h->s.prec == GPT2_BF16
              ? clip_adamw_impl<bf16>(h, lr, beta1, beta2, eps, weight_decay, max_norm, step_t)
              : clip_adamw_impl<float>(h, lr, beta1, beta2, eps, weight_decay, max_norm, step_t);
  if (r != GPT2_OK) return r;
  h->state = ST_IDLE;
  if (h_norm) {
    int st = read_status(h);
    CK(cudaMemcpy(h_norm, h->at<float>(h->p.scalars) + 1, 4, cudaMemcpyDeviceToHost));
    if (st != GPT2_OK) return st;
  }
  return GPT2_OK;
}

}  // extern "C"

namespace {

// Captures the host-buffer step (staging copies in, forward, backward, clip +
// AdamW with device hyperparameters, loss / norm / status out, status cleared)
// into h->host_exec.  Capture runs on a private stream; h->stream is restored.
int build_host_graph(gpt2* h) {
  const size_t bytes = (size_t)h->s.M() * 4;
  if (!h->pin_tok) CK(cudaHostAlloc(reinterpret_cast<void**>(&h->pin_tok), bytes, cudaHostAllocDefault));
  if (!h->pin_tgt) CK(cudaHostAlloc(reinterpret_cast<void**>(&h->pin_tgt), bytes, cudaHostAllocDefault));
  if (!h->pin_hyp) CK(cudaHostAlloc(reinterpret_cast<void**>(&h->pin_hyp), sizeof(OptHyper), cudaHostAllocDefault));
  if (!h->pin_out) CK(cudaHostAlloc(reinterpret_cast<void**>(&h->pin_out), 16, cudaHostAllocDefault));
  if (!h->cap_stream) CK(cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking));
  CK(cudaStreamSynchronize(h->stream));
  const cudaStream_t user = h->stream;
  h->stream = h->cap_stream;
  cudaGraph_t graph = nullptr;
  int r = GPT2_OK;
  cudaError_t e = cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal);
  if (e == cudaSuccess) {
    OptHyper* dh = h->at<OptHyper>(h->p.hyper);
    unsigned* status = h->at<unsigned>(h->p.status);
    cudaMemcpyAsync(h->at<int32_t>(h->p.tokens), h->pin_tok, bytes, cudaMemcpyHostToDevice, h->stream);
    cudaMemcpyAsync(h->at<int32_t>(h->p.targets), h->pin_tgt, bytes, cudaMemcpyHostToDevice, h->stream);
    cudaMemcpyAsync(dh, h->pin_hyp, sizeof(OptHyper), cudaMemcpyHostToDevice, h->stream);
    r = h->s.prec == GPT2_BF16 ? forward_impl<bf16>(h) : forward_impl<float>(h);
    if (r == GPT2_OK) r = h->s.prec == GPT2_BF16 ? backward_impl<bf16>(h) : backward_impl<float>(h);
    if (r == GPT2_OK)
      r = h->s.prec == GPT2_BF16 ? clip_adamw_impl<bf16>(h, 0.f, 0.f, 0.f, 0.f, 0.f, 1.f, 1, dh)
                                 : clip_adamw_impl<float>(h, 0.f, 0.f, 0.f, 0.f, 0.f, 1.f, 1, dh);
    cudaMemcpyAsync(h->pin_out, h->at<float>(h->p.scalars), 8, cudaMemcpyDeviceToHost, h->stream);
    cudaMemcpyAsync(h->pin_out + 2, status, 4, cudaMemcpyDeviceToHost, h->stream);
    cudaMemsetAsync(status, 0, 4, h->stream);
    e = cudaStreamEndCapture(h->cap_stream, &graph);
  }
  h->stream = user;
  if (r == GPT2_OK && e == cudaSuccess) e = cudaGraphInstantiate(&h->host_exec, graph, 0);
  if (graph) cudaGraphDestroy(graph);
  if (r != GPT2_OK) {
    h->host_exec = nullptr;
    return r;
  }
  if (e != cudaSuccess) {
    h->host_exec = nullptr;
    return cuda_fail(e, "gpt2_train_step_host graph");
  }
  return GPT2_OK;
}

}  // namespace

extern "C" {

int gpt2_grad_accumulate(gpt2_t* h, int first, float scale) {
  if (!h) return GPT2_E_INVAL;
  if (h->state != ST_BWD) return GPT2_E_STATE;
  float* acc = h->at<float>(h->p.grad_acc);
  const float* loss = h->at<float>(h->p.scalars);
  float* acc_loss = h->at<float>(h->p.scalars) + 6;
  if (h->s.prec == GPT2_BF16)
    grad_accumulate<bf16>(acc, h->at<bf16>(h->p.grads), (long long)h->N, scale, first ? 1 : 0, loss, acc_loss,
                          h->stream);
  else
    grad_accumulate<float>(acc, h->at<float>(h->p.grads), (long long)h->N, scale, first ? 1 : 0, loss, acc_loss,
                           h->stream);
  CK(cudaGetLastError());
  h->state = ST_ACC;
  return GPT2_OK;
}

int gpt2_clip_adamw_accumulated(gpt2_t* h, float lr, float beta1, float beta2, float eps, float weight_decay,
                                float max_norm, int step_t, float* h_norm) {
  if (!h) return GPT2_E_INVAL;
  if (step_t < 0 || !(max_norm > 0.f)) return GPT2_E_INVAL;
  if (h->state != ST_ACC) return GPT2_E_STATE;
  const float* acc = h->at<float>(h->p.grad_acc);
  int r = h->s.prec == GPT2_BF16
              ? clip_adamw_grads<bf16, float>(h, acc, h->at<float>(h->p.scalars) + 6, lr, beta1, beta2, eps,
                                              weight_decay, max_norm, step_t, nullptr)
              : clip_adamw_grads<float, float>(h, acc, h->at<float>(h->p.scalars) + 6, lr, beta1, beta2, eps,
                                               weight_decay, max_norm, step_t, nullptr);
  if (r != GPT2_OK) return r;
  h->state = ST_IDLE;
  if (h_norm) {
    int st = read_status(h);
    CK(cudaMemcpy(h_norm, h->at<float>(h->p.scalars) + 1, 4, cudaMemcpyDeviceToHost));
    if (st != GPT2_OK) return st;
  }
  return GPT2_OK;
}

int gpt2_train_step_host(gpt2_t* h, const int32_t* h_tokens, const int32_t* h_targets, float lr,
                         float beta1, float beta2, float eps, float weight_decay, float max_norm,
                         int step_t, float* h_loss, float* h_norm) {
  if (!h || !h_tokens || !h_targets) return GPT2_E_INVAL;
  if (step_t < 0 || !(max_norm > 0.f)) return GPT2_E_INVAL;
  const size_t bytes = (size_t)h->s.M() * 4;
  if (h->prof_on) {  // per-region events: run the step eagerly
    int32_t* dt = h->at<int32_t>(h->p.tokens);
    int32_t* dg = h->at<int32_t>(h->p.targets);
    CK(cudaMemcpyAsync(dt, h_tokens, bytes, cudaMemcpyHostToDevice, h->stream));
    CK(cudaMemcpyAsync(dg, h_targets, bytes, cudaMemcpyHostToDevice, h->stream));
    int r = h->s.prec == GPT2_BF16 ? forward_impl<bf16>(h) : forward_impl<float>(h);
    if (r != GPT2_OK) return r;
    h->state = ST_FWD;
    r = gpt2_backward(h);
    if (r != GPT2_OK) return r;
    r = gpt2_clip_adamw(h, lr, beta1, beta2, eps, weight_decay, max_norm, step_t, nullptr);
    if (r != GPT2_OK) return r;
    float sc[2];
    CK(cudaMemcpyAsync(sc, h->at<float>(h->p.scalars), 8, cudaMemcpyDeviceToHost, h->stream));
    int st = read_status(h);
    if (h_loss) *h_loss = sc[0];
    if (h_norm) *h_norm = sc[1];
    return st;
  }
  if (!h->host_exec) {
    int r = build_host_graph(h);
    if (r != GPT2_OK) return r;
  }
  std::memcpy(h->pin_tok, h_tokens, bytes);
  std::memcpy(h->pin_tgt, h_targets, bytes);
  *h->pin_hyp = OptHyper{lr, beta1, beta2, eps, weight_decay, max_norm, step_t, 0};
  CK(cudaGraphLaunch(h->host_exec, h->stream));
  CK(cudaStreamSynchronize(h->stream));
  h->state = ST_IDLE;
  if (h_loss) *h_loss = h->pin_out[0];
  if (h_norm) *h_norm = h->pin_out[1];
  unsigned st;
  std::memcpy(&st, h->pin_out + 2, 4);
  if (st & ST_TIMEOUT) {
    clear_sk_flags(h);
    return GPT2_E_TIMEOUT;
  }
  if (st & ST_TOKEN) return GPT2_E_TOKEN;
  if (st & ST_NONFINITE) return GPT2_E_NONFINITE;
  return GPT2_OK;
}

float gpt2_lr_schedule(int step_t, float max_lr, int warmup_steps, int total_steps, float final_frac) {
  if (step_t < 1 || warmup_steps < 0 || total_steps <= warmup_steps || !(max_lr >= 0.f)) return -1.f;
  if (step_t <= warmup_steps) return (float)((double)max_lr * step_t / warmup_steps);
  double r = (double)(step_t - 1 - warmup_steps) / (double)(total_steps - warmup_steps);
  r = r < 0.0 ? 0.0 : (r > 1.0 ? 1.0 : r);
  const double f = final_frac;
  return (float)((double)max_lr * (f + (1.0 - f) * 0.5 * (1.0 + cos(3.14159265358979323846 * r))));
}

const float* gpt2_device_loss(gpt2_t* h) { return h ? h->at<float>(h->p.scalars) : nullptr; }
const float* gpt2_device_norm(gpt2_t* h) { return h ? h->at<float>(h->p.scalars) + 1 : nullptr; }

int gpt2_sync_status(gpt2_t* h) {
  if (!h) return GPT2_E_INVAL;
  return read_status(h);
}

int gpt2_set_guard(gpt2_t* h, float loss_z, float norm_z, int window) {
  if (!h) return GPT2_E_INVAL;
  if (window < 2 || window > kGuardMaxWindow || !(loss_z == loss_z) || !(norm_z == norm_z)) return GPT2_E_INVAL;
  return reset_guard(h, loss_z, norm_z, window);
}

int gpt2_guard_read(gpt2_t* h, float* z_loss, float* z_norm, int* skipped_spike, int* skipped_nonfinite,
                    int* last_skipped) {
  if (!h) return GPT2_E_INVAL;
  GuardState g;
  CK(cudaStreamSynchronize(h->stream));
  CK(cudaMemcpy(&g, h->at<GuardState>(h->p.guard), offsetof(GuardState, pad), cudaMemcpyDeviceToHost));
  if (z_loss) *z_loss = g.z_loss;
  if (z_norm) *z_norm = g.z_norm;
  if (skipped_spike) *skipped_spike = g.skipped_spike;
  if (skipped_nonfinite) *skipped_nonfinite = g.skipped_nonfinite;
  if (last_skipped) *last_skipped = g.last_skipped;
  return GPT2_OK;
}

const char* gpt2_strerror(int status) {
  switch (status) {
    case GPT2_OK: return "ok";
    case GPT2_E_INVAL: return "invalid argument";
    case GPT2_E_STATE: return "call out of order";
    case GPT2_E_TOKEN: return "token id out of range (clamped)";
    case GPT2_E_CUDA: return "CUDA error";
    case GPT2_E_TIMEOUT: return "bounded wait expired in a pipelined kernel";
    case GPT2_E_NONFINITE: return "non-finite loss or gradient norm";
    case GPT2_E_UNSUPPORTED: return "unsupported shape";
    default: return "unknown status";
  }
}

const char* gpt2_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

// ---------------------------------------------------------------- standalone kernels
static bool al16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int T,
             int d, long long sb, long long sh, long long st, long long osb, long long osh,
             long long ost, float scale, void* stream) {
  if (!al16(q) || !al16(k) || !al16(v) || !al16(o) || !lse) return GPT2_E_INVAL;
  if (B <= 0 || H <= 0 || T <= 0) return GPT2_E_INVAL;
  if (d != 64) return GPT2_E_UNSUPPORTED;
  AttnArgs a;
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
  a.B = B; a.H = H; a.T = T; a.d = d;
  a.sb = sb; a.sh = sh; a.st = st; a.osb = osb; a.osh = osh; a.ost = ost;
  a.scale = scale;
  int e = attn_fwd_tc(a, static_cast<cudaStream_t>(stream));
  if (e == (int)cudaErrorInvalidValue) return GPT2_E_INVAL;
  if (e) return cuda_fail((cudaError_t)e, "attn_fwd");
  return GPT2_OK;
}

size_t attn_workspace_bytes(int B, int H, int T) { return (size_t)B * H * T * sizeof(float); }

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dO, void* dq, void* dk, void* dv, int B, int H, int T, int d, long long sb,
             long long sh, long long st, long long osb, long long osh, long long ost, float scale,
             void* workspace, size_t workspace_bytes, void* stream) {
  if (!al16(q) || !al16(k) || !al16(v) || !al16(o) || !lse || !al16(dO) || !al16(dq) || !al16(dk) ||
      !al16(dv))
    return GPT2_E_INVAL;
  if (B <= 0 || H <= 0 || T <= 0) return GPT2_E_INVAL;
  if (d != 64) return GPT2_E_UNSUPPORTED;
  if (!workspace || workspace_bytes < attn_workspace_bytes(B, H, T)) return GPT2_E_INVAL;
  AttnArgs a;
  a.q = q; a.k = k; a.v = v; a.o = const_cast<void*>(o); a.lse = const_cast<float*>(lse); a.dO = dO;
  a.dq = dq; a.dk = dk; a.dv = dv; a.Dbuf = static_cast<float*>(workspace);
  a.B = B; a.H = H; a.T = T; a.d = d;
  a.sb = sb; a.sh = sh; a.st = st; a.osb = osb; a.osh = osh; a.ost = ost;
  a.scale = scale;
  int e = attn_bwd_bf16(a, static_cast<cudaStream_t>(stream));
  if (e == (int)cudaErrorInvalidValue) return GPT2_E_INVAL;
  if (e) return cuda_fail((cudaError_t)e, "attn_bwd");
  return GPT2_OK;
}

// workspace: logits bf16 [M, Vpad] | pmax, psum f32 [M, tiles] | ztgt, lse, rows f32 [M] | status
static size_t cls_off(int M, int Vpad, int which) {
  const int tiles = (Vpad + gemm_tc_stat_cols() - 1) / gemm_tc_stat_cols();
  size_t cur = 0;
  size_t offs[8];
  offs[0] = take(cur, (size_t)M * Vpad * 2);
  offs[1] = take(cur, (size_t)M * tiles * 4);
  offs[2] = take(cur, (size_t)M * tiles * 4);
  offs[3] = take(cur, (size_t)M * 4);
  offs[4] = take(cur, (size_t)M * 4);
  offs[5] = take(cur, (size_t)M * 4);
  offs[6] = take(cur, 16);
  offs[7] = cur;
  return offs[which];
}

size_t classifier_workspace_bytes(int M, int C, int Vpad) {
  (void)C;
  if (M <= 0 || Vpad <= 0) return 0;
  return cls_off(M, Vpad, 7);
}

int classifier_fwd_bwd(const void* x, const void* w, const int32_t* targets, int M, int C, int V,
                       int Vpad, float* d_loss, void* dx, void* dw, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (!al16(x) || !al16(w) || !targets || !d_loss || !al16(dx) || !al16(dw) || !workspace)
    return GPT2_E_INVAL;
  if (M <= 0 || C <= 0 || V <= 0 || Vpad < V || C % 8 || Vpad % 8) return GPT2_E_INVAL;
  if (workspace_bytes < classifier_workspace_bytes(M, C, Vpad) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255))
    return GPT2_E_INVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  bf16* logits = reinterpret_cast<bf16*>(ws + cls_off(M, Vpad, 0));
  float* pmax = reinterpret_cast<float*>(ws + cls_off(M, Vpad, 1));
  float* psum = reinterpret_cast<float*>(ws + cls_off(M, Vpad, 2));
  float* ztgt = reinterpret_cast<float*>(ws + cls_off(M, Vpad, 3));
  float* lse = reinterpret_cast<float*>(ws + cls_off(M, Vpad, 4));
  float* rows = reinterpret_cast<float*>(ws + cls_off(M, Vpad, 5));
  unsigned* status = reinterpret_cast<unsigned*>(ws + cls_off(M, Vpad, 6));
  const int tiles = (Vpad + gemm_tc_stat_cols() - 1) / gemm_tc_stat_cols();
  GemmArgs g;
  g.A = x; g.lda = C; g.B = w; g.ldb = C; g.M = M; g.N = Vpad; g.K = C;
  g.epi = EPI_CE; g.D = logits; g.ldd = Vpad;
  g.ce_max = pmax; g.ce_sum = psum; g.ce_ld = tiles; g.ce_tgt = ztgt; g.targets = targets; g.V = V;
  int e = gemm_tc(g, 1, nullptr, 0, status, st);
  if (e) return cuda_fail((cudaError_t)e, "classifier logits");
  ce_reduce_partials(pmax, psum, tiles, tiles, ztgt, M, lse, rows, st);
  mean_reduce(d_loss, rows, M, status, st);
  ce_dlogits<bf16>(logits, Vpad, lse, targets, M, V, Vpad, 1.0f / (float)M, st);
  g = GemmArgs();
  g.A = logits; g.lda = Vpad; g.B = w; g.ldb = C; g.b_mn = 1;
  g.M = M; g.N = C; g.K = Vpad; g.D = dx; g.ldd = C;
  e = gemm_tc(g, 1, nullptr, 0, status, st);
  if (e) return cuda_fail((cudaError_t)e, "classifier dx");
  g = GemmArgs();
  g.A = logits; g.lda = Vpad; g.a_mn = 1; g.B = x; g.ldb = C; g.b_mn = 1;
  g.M = Vpad; g.N = C; g.K = M; g.D = dw; g.ldd = C;
  e = gemm_tc(g, 1, nullptr, 0, status, st);
  if (e) return cuda_fail((cudaError_t)e, "classifier dw");
  cudaError_t ce = cudaGetLastError();
  if (ce != cudaSuccess) return cuda_fail(ce, "classifier_fwd_bwd");
  return GPT2_OK;
}

int gpt2_encoder_fwd(const int32_t* tok, const void* wte, const void* wpe, void* x0, int B, int T,
                     int C, int V, int precision, void* d_status, void* stream) {
  if (!tok || !al16(wte) || !al16(wpe) || !al16(x0)) return GPT2_E_INVAL;
  if (B <= 0 || T <= 0 || C <= 0 || C % 8 || V <= 0) return GPT2_E_INVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* status = static_cast<unsigned*>(d_status);
  if (precision == GPT2_BF16)
    encoder_fwd<bf16>(static_cast<bf16*>(x0), tok, static_cast<const bf16*>(wte),
                      static_cast<const bf16*>(wpe), B, T, C, V, status, st);
  else if (precision == GPT2_FP32)
    encoder_fwd<float>(static_cast<float*>(x0), tok, static_cast<const float*>(wte),
                       static_cast<const float*>(wpe), B, T, C, V, status, st);
  else
    return GPT2_E_INVAL;
  CK(cudaGetLastError());
  return GPT2_OK;
}

int gpt2_encoder_bwd(const int32_t* tok, float* dx0, void* dwte, void* dwpe, int B, int T,
                     int C, int V, int precision, void* workspace, size_t workspace_bytes,
                     void* stream) {
  if (!tok || !al16(dx0) || !dwte || !dwpe || !workspace) return GPT2_E_INVAL;
  if (B <= 0 || T <= 0 || C <= 0 || C % 8 || V <= 0) return GPT2_E_INVAL;
  if ((long long)B * T > 16384) return GPT2_E_UNSUPPORTED;
  if (workspace_bytes < (size_t)8 * B * T) return GPT2_E_INVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* order = static_cast<uint32_t*>(workspace);
  sort_tokens(order, tok, B * T, V, st);
  if (precision == GPT2_BF16)
    encoder_bwd<bf16>(static_cast<bf16*>(dwte), static_cast<bf16*>(dwpe), dx0, order, tok, B, T, C, st);
  else if (precision == GPT2_FP32)
    encoder_bwd<float>(static_cast<float*>(dwte), static_cast<float*>(dwpe), dx0, order, tok, B, T, C, st);
  else
    return GPT2_E_INVAL;
  CK(cudaGetLastError());
  return GPT2_OK;
}

int gemm_bf16(const void* A, const void* B, void* D, int M, int N, int K, long long lda,
              long long ldb, long long ldd, int a_mn, int b_mn, int d_f32, int splits,
              void* workspace, size_t workspace_bytes, void* stream) {
  if (!al16(A) || !al16(B) || !al16(D)) return GPT2_E_INVAL;
  if (M <= 0 || N <= 0 || K <= 0 || N % 8 || lda % 8 || ldb % 8 || ldd % 8) return GPT2_E_INVAL;
  GemmArgs g;
  g.A = A; g.lda = lda; g.a_mn = a_mn ? 1 : 0; g.B = B; g.ldb = ldb; g.b_mn = b_mn ? 1 : 0;
  g.M = M; g.N = N; g.K = K; g.D = D; g.ldd = ldd; g.epi = d_f32 ? EPI_F32 : EPI_STORE;
  if (splits < -2) return GPT2_E_INVAL;
  if (splits < 0) {
    if (!al16(workspace) || workspace_bytes < gemm_tc_sk_ws_bytes()) return GPT2_E_INVAL;
  } else {
    if (splits == 0) splits = gemm_tc_pick_splits(M, N, K, gemm_tc_pairs());
    if (splits > 1 && workspace_bytes < gemm_tc_ws_bytes(M, N, splits)) return GPT2_E_INVAL;
  }
  int e = gemm_tc(g, splits, workspace, workspace_bytes, nullptr, static_cast<cudaStream_t>(stream));
  if (e == (int)cudaErrorInvalidValue) return GPT2_E_INVAL;
  if (e) return cuda_fail((cudaError_t)e, "gemm_bf16");
  return GPT2_OK;
}

size_t gemm_bf16_sk_workspace_bytes(void) { return gemm_tc_sk_ws_bytes(); }

int gemm_bf16_pairs(void) { return gemm_tc_pairs(); }

int gemm_bf16_epilogue(const void* A, const void* B, void* D, void* D2, const void* bias, const void* X,
                       float* colpart, int M, int N, int K, long long lda, long long ldb, long long ldd,
                       int a_mn, int b_mn, int epi, int splits, void* workspace, size_t workspace_bytes,
                       void* stream) {
  if (epi < 1 || epi > 4) return GPT2_E_INVAL;
  if (!al16(A) || !al16(B) || !al16(D)) return GPT2_E_INVAL;
  if (M <= 0 || N <= 0 || K <= 0 || N % 8 || lda % 8 || ldb % 8 || ldd % 8) return GPT2_E_INVAL;
  if (epi != 4 && !al16(bias)) return GPT2_E_INVAL;
  if ((epi == 2 || epi == 4) && !al16(X)) return GPT2_E_INVAL;
  if (epi == 3 && !al16(D2)) return GPT2_E_INVAL;
  if (splits < -2 || splits > 1) return GPT2_E_INVAL;
  if (splits < 0 && (!al16(workspace) || workspace_bytes < gemm_tc_sk_ws_bytes())) return GPT2_E_INVAL;
  GemmArgs g;
  g.A = A; g.lda = lda; g.a_mn = a_mn ? 1 : 0; g.B = B; g.ldb = ldb; g.b_mn = b_mn ? 1 : 0;
  g.M = M; g.N = N; g.K = K; g.D = D; g.ldd = ldd;
  g.epi = epi == 1 ? EPI_BIAS : epi == 2 ? EPI_BIAS_RESID : epi == 3 ? EPI_BIAS_GELU : EPI_GELU_BWD;
  g.bias = bias; g.D2 = D2; g.resid = X; g.ldr = ldd; g.aux = X; g.ldaux = ldd;
  if (epi == 4) g.colpart = colpart;
  int e = gemm_tc(g, splits == 0 ? 1 : splits, workspace, workspace_bytes, nullptr,
                  static_cast<cudaStream_t>(stream));
  if (e == (int)cudaErrorInvalidValue) return GPT2_E_INVAL;
  if (e) return cuda_fail((cudaError_t)e, "gemm_bf16_epilogue");
  return GPT2_OK;
}

int gpt2_test_set_gemm_poison(int on) {
  const int old = g_test_poison;
  g_test_poison = on ? (old | POISON_GEMM_TMA) : (old & ~POISON_GEMM_TMA);
  return (old & POISON_GEMM_TMA) ? 1 : 0;
}

int gpt2_test_set_poison(int mask) {
  const int old = g_test_poison;
  g_test_poison = mask;
  return old;
}

int gemm_bf16_status(const void* A, const void* B, void* D, int M, int N, int K, long long lda,
                     long long ldb, long long ldd, int a_mn, int b_mn, int splits, void* workspace,
                     size_t workspace_bytes, void* d_status_word, void* stream) {
  if (!al16(A) || !al16(B) || !al16(D) || !d_status_word) return GPT2_E_INVAL;
  if (splits != 1 && splits != -1 && splits != -2) return GPT2_E_INVAL;
  if (splits < 0 && (!al16(workspace) || workspace_bytes < gemm_tc_sk_ws_bytes())) return GPT2_E_INVAL;
  GemmArgs g;
  g.A = A; g.lda = lda; g.a_mn = a_mn ? 1 : 0; g.B = B; g.ldb = ldb; g.b_mn = b_mn ? 1 : 0;
  g.M = M; g.N = N; g.K = K; g.D = D; g.ldd = ldd; g.epi = EPI_STORE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* status = static_cast<unsigned*>(d_status_word);
  CK(cudaMemsetAsync(status, 0, 4, st));
  int e = gemm_tc(g, splits, splits < 0 ? workspace : nullptr, splits < 0 ? workspace_bytes : 0, status, st);
  if (e == (int)cudaErrorInvalidValue) return GPT2_E_INVAL;
  if (e) return cuda_fail((cudaError_t)e, "gemm_bf16_status");
  unsigned hs = 0;
  CK(cudaStreamSynchronize(st));
  CK(cudaMemcpy(&hs, status, 4, cudaMemcpyDeviceToHost));
  if (hs & ST_TIMEOUT) return GPT2_E_TIMEOUT;
  return GPT2_OK;
}

}  // extern "C"
