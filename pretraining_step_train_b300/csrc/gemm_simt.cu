// fp32 GEMM on CUDA cores for the fp32 parity mode of the step.
//
// D[m, n] = sum_k A(m, k) B(n, k) with either operand K-major or MN-major,
// 64x64 output tiles, 4x4 outputs per thread, fp32 FMA accumulation, and the
// same epilogues as the tensor-core path (bias, residual, GELU, GELU').
#include "common.cuh"
#include "internal.h"

namespace gpt2k {

constexpr int SB_M = 64, SB_N = 64, SB_K = 16;

__global__ void __launch_bounds__(256) k_gemm_simt(GemmArgs g) {
  pdl_begin();
  __shared__ float As[SB_K][SB_M + 4];
  __shared__ float Bs[SB_K][SB_N + 4];
  const float* A = static_cast<const float*>(g.A);
  const float* B = static_cast<const float*>(g.B);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * SB_M, n0 = blockIdx.x * SB_N;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < g.K; k0 += SB_K) {
    for (int i = threadIdx.x; i < SB_M * SB_K; i += 256) {
      int mm, kk;
      if (!g.a_mn) { mm = i / SB_K; kk = i % SB_K; } else { kk = i / SB_M; mm = i % SB_M; }
      int gm = m0 + mm, gk = k0 + kk;
      float v = 0.f;
      if (gm < g.M && gk < g.K) v = g.a_mn ? A[(long long)gk * g.lda + gm] : A[(long long)gm * g.lda + gk];
      As[kk][mm] = v;
    }
    for (int i = threadIdx.x; i < SB_N * SB_K; i += 256) {
      int nn, kk;
      if (!g.b_mn) { nn = i / SB_K; kk = i % SB_K; } else { kk = i / SB_N; nn = i % SB_N; }
      int gn = n0 + nn, gk = k0 + kk;
      float v = 0.f;
      if (gn < g.N && gk < g.K) v = g.b_mn ? B[(long long)gk * g.ldb + gn] : B[(long long)gn * g.ldb + gk];
      Bs[kk][nn] = v;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SB_K; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* D = static_cast<float*>(g.D);
  const float* bias = static_cast<const float*>(g.bias);
  const float* resid = static_cast<const float*>(g.resid);
  const float* aux = static_cast<const float*>(g.aux);
  float* D2 = static_cast<float*>(g.D2);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= g.N) continue;
      float v = acc[i][j];
      const long long o = (long long)m * g.ldd + n;
      switch (g.epi) {
        case EPI_BIAS: v += bias[n]; break;
        case EPI_BIAS_RESID: v += bias[n] + resid[(long long)m * g.ldr + n]; break;
        case EPI_BIAS_GELU: v += bias[n]; D2[o] = gelu_f(v); v = gelu_grad_f(v); break;
        case EPI_GELU_BWD: v *= aux[(long long)m * g.ldaux + n]; break;
        case EPI_BIAS_GELU_H: v += bias[n]; D2[o] = gelu_f(v); break;
        case EPI_GELU_BWD_H: v *= gelu_grad_f(aux[(long long)m * g.ldaux + n]); break;
        default: break;
      }
      D[o] = v;
    }
  }
}

int gemm_simt(const GemmArgs& g, cudaStream_t s) {
  if (g.epi == EPI_CE) return (int)cudaErrorInvalidValue;
  dim3 grid((g.N + SB_N - 1) / SB_N, (g.M + SB_M - 1) / SB_M);
  launch_k(k_gemm_simt, grid, 256, 0, s, g);
  return (int)cudaGetLastError();
}

}  // namespace gpt2k
