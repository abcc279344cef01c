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
// on the first call made on a device, with that device current, and cached
// together with the id of the context it belongs to; a call in a new context
// (after a device reset) looks it up again.  The first call on a device should
// therefore be made before any stream capture.  Every call on a device uses
// the same array: calls whose kernels may overlap on the GPU (different
// streams, no ordering between them) race on it.  The array keeps whatever the
// last call left in it; nothing needs clearing, because the dQ kernel, which
// runs first, writes every row of D before the dK/dV kernel reads it.
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "../../include/gpt2.h"

static __device__ __align__(256) float g_attn_bwd_scratch[ATTN_BWD_NOALLOC_MAX_ROWS];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
struct CachedAddress {
  unsigned long long ctx = 0;  // id of the context the address belongs to (0: none cached)
  float* ptr = nullptr;
};
CachedAddress g_scratch[kMaxDevices];

// Device address of g_attn_bwd_scratch in the current device's current context.
cudaError_t scratch_for_current_device(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const unsigned long long id = gpt2k::current_context_id();
  if (id == 0 || g_scratch[dev].ctx != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_bwd_scratch);  // makes the device's context current if it was not
    if (e != cudaSuccess) return e;
    g_scratch[dev].ptr = static_cast<float*>(p);
    g_scratch[dev].ctx = gpt2k::current_context_id();
  }
  *out = g_scratch[dev].ptr;
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
  cudaError_t ce = scratch_for_current_device(&scratch);
  if (ce != cudaSuccess) return gpt2k::cuda_fail(ce, "attn_bwd_noalloc: scratch address");
  gpt2k::AttnArgs a;
  a.q = q; a.k = k; a.v = v; a.o = const_cast<void*>(o); a.lse = const_cast<float*>(lse); a.dO = dO;
  a.dq = dq; a.dk = dk; a.dv = dv; a.Dbuf = scratch;
  a.B = B; a.H = H; a.T = T; a.d = d;
  a.sb = sb; a.sh = sh; a.st = st; a.osb = osb; a.osh = osh; a.ost = ost;
  a.scale = scale;
  int e = gpt2k::attn_bwd_bf16(a, static_cast<cudaStream_t>(stream));
  if (e == (int)cudaErrorInvalidValue) return GPT2_E_INVAL;
  if (e) return gpt2k::cuda_fail((cudaError_t)e, "attn_bwd_noalloc");
  return GPT2_OK;
}
