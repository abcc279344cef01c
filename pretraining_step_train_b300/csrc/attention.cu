// Causal multi-head attention, forward and backward, never materialising the
// T x T score matrix (online softmax over key tiles, FlashAttention-style;
// "Let's reproduce GPT-2 (124M)" wiki page, "GPU optimisation ladder":
// FlashAttention gives the same result without storing T x T).
//
// bf16 path (d = 64): the tcgen05 kernels of attention_tc.cu; this file adds
// the backward's pre-pass D = rowsum(dO * O).
//
// fp32 path: one warp per query (or key) row on CUDA cores, for the fp32
// parity mode.
//
// Layout: element (b, h, t, i) of q/k/v/dq/dk/dv sits at b*sb + h*sh + t*st + i,
// of o/dO at b*osb + h*osh + t*ost + i; lse and D are [B, H, T] fp32 with lse
// in natural log.  Causal mask keeps keys j <= query i.
#include "common.cuh"
#include "internal.h"

#include <math.h>

namespace gpt2k {


// ------------------------------------------------------------------ backward pre-pass
// D[b, h, i] = sum_c dO[i, c] * O[i, c]   (one warp per row)
template <typename T>
__global__ void k_attn_rowdot(AttnArgs a) {
  pdl_begin();
  const long long row = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= (long long)a.B * a.H * a.T) return;
  const int i = (int)(row % a.T);
  const int bh = (int)(row / a.T);
  const int b = bh / a.H, h = bh % a.H;
  const T* O = static_cast<const T*>(a.o) + b * a.osb + h * a.osh + (long long)i * a.ost;
  const T* dO = static_cast<const T*>(a.dO) + b * a.osb + h * a.osh + (long long)i * a.ost;
  float s = 0.f;
  for (int c = lane; c < a.d; c += 32) s += to_f(O[c]) * to_f(dO[c]);
  s = warp_sum(s);
  if (lane == 0) a.Dbuf[row] = s;
}

static bool strides_ok(const AttnArgs& a) {
  return a.d == 64 && a.st % 8 == 0 && a.sh % 8 == 0 && a.sb % 8 == 0 && a.ost % 8 == 0 &&
         a.osh % 8 == 0 && a.osb % 8 == 0;
}

// bf16: the tcgen05 kernels, which form D = rowsum(dO * O) themselves (into a.Dbuf).
int attn_bwd_bf16(const AttnArgs& a, cudaStream_t s) {
  if (!strides_ok(a)) return (int)cudaErrorInvalidValue;
  return attn_bwd_tc(a, s);
}

// ------------------------------------------------------------------ fp32 (CUDA cores)
// One warp per query row; each lane takes keys j = lane, lane+32, ...; online
// softmax across 32-key chunks; lanes own output columns c = lane, lane+32, ...
constexpr int kF32MaxD = 128;

__global__ void k_attn_fwd_f32(AttnArgs a) {
  pdl_begin();
  const long long row = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= (long long)a.B * a.H * a.T) return;
  const int i = (int)(row % a.T), bh = (int)(row / a.T), b = bh / a.H, h = bh % a.H;
  const long long off = b * a.sb + h * a.sh;
  const float* Q = static_cast<const float*>(a.q) + off + (long long)i * a.st;
  const float* K = static_cast<const float*>(a.k) + off;
  const float* Vp = static_cast<const float*>(a.v) + off;
  const int d = a.d;
  float o[kF32MaxD / 32];
#pragma unroll
  for (int u = 0; u < kF32MaxD / 32; ++u) o[u] = 0.f;
  float m = -INFINITY, l = 0.f;
  for (int j0 = 0; j0 <= i; j0 += 32) {
    const int j = j0 + lane;
    float sj = -INFINITY;
    if (j <= i) {
      float acc = 0.f;
      const float* kr = K + (long long)j * a.st;
      for (int c = 0; c < d; ++c) acc = fmaf(Q[c], kr[c], acc);
      sj = acc * a.scale;
    }
    const float mx = warp_max(sj);
    const float mnew = fmaxf(m, mx);
    const float corr = expf(m - mnew);
    const float p = (j <= i) ? expf(sj - mnew) : 0.f;
    l = l * corr + warp_sum(p);
#pragma unroll
    for (int u = 0; u < kF32MaxD / 32; ++u) o[u] *= corr;
    const int nj = min(32, i - j0 + 1);
    for (int jj = 0; jj < nj; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
      const float* vr = Vp + (long long)(j0 + jj) * a.st;
#pragma unroll
      for (int u = 0; u < kF32MaxD / 32; ++u) {
        int c = lane + u * 32;
        if (c < d) o[u] = fmaf(pj, vr[c], o[u]);
      }
    }
    m = mnew;
  }
  float* O = static_cast<float*>(a.o) + b * a.osb + h * a.osh + (long long)i * a.ost;
#pragma unroll
  for (int u = 0; u < kF32MaxD / 32; ++u) {
    int c = lane + u * 32;
    if (c < d) O[c] = o[u] / l;
  }
  if (lane == 0) a.lse[row] = m + logf(l);
}

// dQ: warp per query row i.
__global__ void k_attn_bwd_dq_f32(AttnArgs a) {
  pdl_begin();
  const long long row = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= (long long)a.B * a.H * a.T) return;
  const int i = (int)(row % a.T), bh = (int)(row / a.T), b = bh / a.H, h = bh % a.H;
  const long long off = b * a.sb + h * a.sh, ooff = b * a.osb + h * a.osh;
  const float* Q = static_cast<const float*>(a.q) + off + (long long)i * a.st;
  const float* dO = static_cast<const float*>(a.dO) + ooff + (long long)i * a.ost;
  const float* K = static_cast<const float*>(a.k) + off;
  const float* Vp = static_cast<const float*>(a.v) + off;
  const float L = a.lse[row], Dr = a.Dbuf[row];
  const int d = a.d;
  float dq[kF32MaxD / 32];
#pragma unroll
  for (int u = 0; u < kF32MaxD / 32; ++u) dq[u] = 0.f;
  for (int j0 = 0; j0 <= i; j0 += 32) {
    const int j = j0 + lane;
    float ds = 0.f;
    if (j <= i) {
      float s = 0.f, dp = 0.f;
      const float* kr = K + (long long)j * a.st;
      const float* vr = Vp + (long long)j * a.st;
      for (int c = 0; c < d; ++c) {
        s = fmaf(Q[c], kr[c], s);
        dp = fmaf(dO[c], vr[c], dp);
      }
      const float p = expf(s * a.scale - L);
      ds = p * (dp - Dr);
    }
    const int nj = min(32, i - j0 + 1);
    for (int jj = 0; jj < nj; ++jj) {
      const float dsj = __shfl_sync(0xffffffffu, ds, jj);
      const float* kr = K + (long long)(j0 + jj) * a.st;
#pragma unroll
      for (int u = 0; u < kF32MaxD / 32; ++u) {
        int c = lane + u * 32;
        if (c < d) dq[u] = fmaf(dsj, kr[c], dq[u]);
      }
    }
  }
  float* dQ = static_cast<float*>(a.dq) + off + (long long)i * a.st;
#pragma unroll
  for (int u = 0; u < kF32MaxD / 32; ++u) {
    int c = lane + u * 32;
    if (c < d) dQ[c] = dq[u] * a.scale;
  }
}

// dK, dV: warp per key row j, lanes over queries i >= j.
__global__ void k_attn_bwd_dkdv_f32(AttnArgs a) {
  pdl_begin();
  const long long row = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= (long long)a.B * a.H * a.T) return;
  const int j = (int)(row % a.T), bh = (int)(row / a.T), b = bh / a.H, h = bh % a.H;
  const long long off = b * a.sb + h * a.sh, ooff = b * a.osb + h * a.osh;
  const float* Q = static_cast<const float*>(a.q) + off;
  const float* dO = static_cast<const float*>(a.dO) + ooff;
  const float* kr = static_cast<const float*>(a.k) + off + (long long)j * a.st;
  const float* vr = static_cast<const float*>(a.v) + off + (long long)j * a.st;
  const float* lse = a.lse + (long long)bh * a.T;
  const float* Dv = a.Dbuf + (long long)bh * a.T;
  const int d = a.d, T = a.T;
  float dk[kF32MaxD / 32], dv[kF32MaxD / 32];
#pragma unroll
  for (int u = 0; u < kF32MaxD / 32; ++u) dk[u] = dv[u] = 0.f;
  for (int i0 = j; i0 < T; i0 += 32) {
    const int i = i0 + lane;
    float p = 0.f, ds = 0.f;
    if (i < T) {
      float s = 0.f, dp = 0.f;
      const float* qr = Q + (long long)i * a.st;
      const float* dor = dO + (long long)i * a.ost;
      for (int c = 0; c < d; ++c) {
        s = fmaf(qr[c], kr[c], s);
        dp = fmaf(dor[c], vr[c], dp);
      }
      p = expf(s * a.scale - lse[i]);
      ds = p * (dp - Dv[i]);
    }
    const int ni = min(32, T - i0);
    for (int ii = 0; ii < ni; ++ii) {
      const float pi = __shfl_sync(0xffffffffu, p, ii);
      const float dsi = __shfl_sync(0xffffffffu, ds, ii);
      const float* qr = Q + (long long)(i0 + ii) * a.st;
      const float* dor = dO + (long long)(i0 + ii) * a.ost;
#pragma unroll
      for (int u = 0; u < kF32MaxD / 32; ++u) {
        int c = lane + u * 32;
        if (c < d) {
          dv[u] = fmaf(pi, dor[c], dv[u]);
          dk[u] = fmaf(dsi, qr[c], dk[u]);
        }
      }
    }
  }
  float* dK = static_cast<float*>(a.dk) + off + (long long)j * a.st;
  float* dV = static_cast<float*>(a.dv) + off + (long long)j * a.st;
#pragma unroll
  for (int u = 0; u < kF32MaxD / 32; ++u) {
    int c = lane + u * 32;
    if (c < d) {
      dK[c] = dk[u] * a.scale;
      dV[c] = dv[u];
    }
  }
}

int attn_fwd_f32(const AttnArgs& a, cudaStream_t s) {
  if (a.d > kF32MaxD) return (int)cudaErrorInvalidValue;
  long long rows = (long long)a.B * a.H * a.T;
  launch_k(k_attn_fwd_f32, (unsigned)((rows * 32 + 255) / 256), 256, 0, s, a);
  return (int)cudaGetLastError();
}

int attn_bwd_f32(const AttnArgs& a, cudaStream_t s) {
  if (a.d > kF32MaxD) return (int)cudaErrorInvalidValue;
  long long rows = (long long)a.B * a.H * a.T;
  unsigned grid = (unsigned)((rows * 32 + 255) / 256);
  launch_k(k_attn_rowdot<float>, grid, 256, 0, s, a);
  launch_k(k_attn_bwd_dq_f32, grid, 256, 0, s, a);
  launch_k(k_attn_bwd_dkdv_f32, grid, 256, 0, s, a);
  return (int)cudaGetLastError();
}

}  // namespace gpt2k
