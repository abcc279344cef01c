// attn_bwd_noalloc: the causal attention backward without a caller-supplied
// workspace (see include/gpt2.h).
//
// Some callers cannot allocate device memory for a workspace: a host runtime
// that has handed the whole device to its own memory pool and forbids library
// allocations, or a latency-critical loop that cannot afford cudaMalloc's
// implicit device synchronisation.  For them the one scratch buffer the
// attention backward needs (the per-row D = rowsum(dO * O), fp32 [B, H, T])
// lives in a fixed-size array in the library's own device memory instead.
//
// The array is static device memory of this library: every GPU that loads the
// library holds it (4 MiB) until the process exits.  Its address is looked up
// once per device, on the first call made with that device current, and
// cached.  That first call should therefore be made before any stream capture.
// Every call on a device uses the same array: calls whose kernels may overlap
// on the GPU (different streams, no ordering between them) race on it.  The
// array keeps whatever the last call left in it; nothing needs clearing,
// because the pre-pass writes every row of D before the dK/dV and dQ kernels
// read it.
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "../../include/gpt2.h"

static __device__ __align__(256) float g_attn_bwd_scratch[ATTN_BWD_NOALLOC_MAX_ROWS];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_attn_bwd_scratch on the current device (looked up once).
cudaError_t scratch_for_current_device(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_bwd_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                                int H, int T, int d, long long sb, long long sh, long long st,
                                long long osb, long long osh, long long ost, float scale,
                                void* stream) {
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !lse || !aligned16(dO) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return GPT2_E_INVAL;
  if (B <= 0 || H <= 0 || T <= 0) return GPT2_E_INVAL;
  if (d != 64) return GPT2_E_UNSUPPORTED;
  if ((long long)B * H * T > ATTN_BWD_NOALLOC_MAX_ROWS) return GPT2_E_UNSUPPORTED;
  float* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return GPT2_E_CUDA;
  gpt2k::AttnArgs a;
  a.q = q; a.k = k; a.v = v; a.o = const_cast<void*>(o); a.lse = const_cast<float*>(lse); a.dO = dO;
  a.dq = dq; a.dk = dk; a.dv = dv; a.Dbuf = scratch;
  a.B = B; a.H = H; a.T = T; a.d = d;
  a.sb = sb; a.sh = sh; a.st = st; a.osb = osb; a.osh = osh; a.ost = ost;
  a.scale = scale;
  int e = gpt2k::attn_bwd_bf16(a, static_cast<cudaStream_t>(stream));
  if (e == (int)cudaErrorInvalidValue) return GPT2_E_INVAL;
  if (e) return GPT2_E_CUDA;
  return GPT2_OK;
}
