// Memory-bound kernels of the GPT-2 step: encoder, LayerNorm, GELU, residual,
// bias-gradient column sums, cross-entropy pieces, fixed-order encoder
// backward, split-K reduction, global gradient norm and AdamW.
//
// All of them stream 16-byte vectors (4 fp32 or 8 bf16 per access) with
// consecutive threads on consecutive addresses, reduce with warp shuffles,
// and keep every reduction in a fixed order so results are bitwise
// reproducible run to run.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

#include <math.h>

namespace gpt2k {

static inline int grid_for(long long work, int block, int cap = 148 * 16) {
  long long g = (work + block - 1) / block;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return (int)g;
}

// ------------------------------------------------------------------ encoder
// x0[b, t, :] = wte[tok[b, t], :] + wpe[t, :]   (one fp32 add, then one rounding)
template <typename T>
__global__ void k_encoder_fwd(T* __restrict__ x0, const int32_t* __restrict__ tok,
                              const T* __restrict__ wte, const T* __restrict__ wpe, int M, int Tn,
                              int C, int V, unsigned* status) {
  pdl_begin();
  constexpr int N = V16<T>::N;
  const int cv = C / N;
  const long long nvec = (long long)M * cv;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < nvec;
       i += (long long)gridDim.x * blockDim.x) {
    int m = (int)(i / cv), c = (int)(i % cv) * N;
    int t = m % Tn;
    int id = tok[m];
    if (id < 0 || id >= V) {
      if (status) atomicOr(status, ST_TOKEN);
      id = 0;
    }
    float a[N], b[N];
    load16(wte + (long long)id * C + c, a);
    load16(wpe + (long long)t * C + c, b);
#pragma unroll
    for (int j = 0; j < N; ++j) a[j] = a[j] + b[j];
    store16(x0 + (long long)m * C + c, a);
  }
}

template <typename T>
void encoder_fwd(T* x0, const int32_t* tok, const T* wte, const T* wpe, int B, int Tn, int C, int V,
                 unsigned* status, cudaStream_t s) {
  long long nvec = (long long)B * Tn * C / V16<T>::N;
  launch_k(k_encoder_fwd<T>, grid_for(nvec, 256), 256, 0, s, x0, tok, wte, wpe, B * Tn, Tn, C, V, status);
}

// Clamp ids outside [0, V) to 0 in place and latch ST_TOKEN.
__global__ void k_check_ids(int32_t* __restrict__ ids, int n, int V, unsigned* status) {
  pdl_begin();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    int t = ids[i];
    if (t < 0 || t >= V) {
      ids[i] = 0;
      if (status) atomicOr(status, ST_TOKEN);
    }
  }
}
void check_ids(int32_t* ids, int n, int V, unsigned* status, cudaStream_t s) {
  launch_k(k_check_ids, grid_for(n, 256, 148), 256, 0, s, ids, n, V, status);
}

// ------------------------------------------------------------------ LayerNorm forward
// Each warp normalises two rows; both rows are loaded up front and stay in
// registers in their storage format (16-byte vectors: packed bf16 or fp32),
// unpacked on each of the three passes (mean, biased variance, output), so a
// lane keeps 2 * MAXV loads in flight and a launch fits in about one wave.
template <typename T>
__device__ __forceinline__ void unpack16(const uint4& u, float* out) {
  if constexpr (sizeof(T) == 4) {
    out[0] = __uint_as_float(u.x); out[1] = __uint_as_float(u.y);
    out[2] = __uint_as_float(u.z); out[3] = __uint_as_float(u.w);
  } else {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      out[2 * i] = __uint_as_float(w[i] << 16);
      out[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}

constexpr int kLnfRows = 2;  // rows per warp

template <typename T, int MAXV>
__global__ void __launch_bounds__(256) k_layernorm_fwd(T* __restrict__ y, float* __restrict__ mean,
                                                       float* __restrict__ rstd, const T* __restrict__ x,
                                                       const T* __restrict__ w, const T* __restrict__ b,
                                                       int M, int C) {
  pdl_begin();
  constexpr int N = V16<T>::N;
  const int row0 = ((blockIdx.x * blockDim.x + threadIdx.x) >> 5) * kLnfRows;
  const int lane = threadIdx.x & 31;
  if (row0 >= M) return;
  const int nv = C / N;
  uint4 raw[kLnfRows][MAXV];
#pragma unroll
  for (int rr = 0; rr < kLnfRows; ++rr) {
    const T* xr = x + (long long)(row0 + rr) * C;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
      const int vi = lane + j * 32;
      if (row0 + rr < M && vi < nv) raw[rr][j] = *reinterpret_cast<const uint4*>(xr + vi * N);
    }
  }
#pragma unroll
  for (int rr = 0; rr < kLnfRows; ++rr) {
    const int row = row0 + rr;
    if (row >= M) break;
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
      if (lane + j * 32 < nv) {
        float v[N];
        unpack16<T>(raw[rr][j], v);
#pragma unroll
        for (int e = 0; e < N; ++e) s += v[e];
      }
    }
    s = warp_sum(s);
    const float mu = s / (float)C;
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
      if (lane + j * 32 < nv) {
        float v[N];
        unpack16<T>(raw[rr][j], v);
#pragma unroll
        for (int e = 0; e < N; ++e) {
          const float d = v[e] - mu;
          ss += d * d;
        }
      }
    }
    ss = warp_sum(ss);
    const float rs = 1.0f / sqrtf(ss / (float)C + 1e-5f);
    T* yr = y + (long long)row * C;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
      const int vi = lane + j * 32;
      if (vi < nv) {
        float v[N], wv[N], bv[N], o[N];
        unpack16<T>(raw[rr][j], v);
        load16(w + vi * N, wv);
        load16(b + vi * N, bv);
#pragma unroll
        for (int e = 0; e < N; ++e) o[e] = (v[e] - mu) * rs * wv[e] + bv[e];
        store16(yr + vi * N, o);
      }
    }
    if (lane == 0) {
      mean[row] = mu;
      rstd[row] = rs;
    }
  }
}

template <typename T>
void layernorm_fwd(T* y, float* mean, float* rstd, const T* x, const T* w, const T* b, int M, int C,
                   cudaStream_t s) {
  const int nv = C / V16<T>::N;
  const int per = (nv + 31) / 32;
  const int block = 256;
  const long long warps = (M + kLnfRows - 1) / kLnfRows;
  const int grid = (int)((warps * 32 + block - 1) / block);
  if (per <= 1) launch_k(k_layernorm_fwd<T, 1>, grid, block, 0, s, y, mean, rstd, x, w, b, M, C);
  else if (per <= 2) launch_k(k_layernorm_fwd<T, 2>, grid, block, 0, s, y, mean, rstd, x, w, b, M, C);
  else if (per <= 3) launch_k(k_layernorm_fwd<T, 3>, grid, block, 0, s, y, mean, rstd, x, w, b, M, C);
  else if (per <= 4) launch_k(k_layernorm_fwd<T, 4>, grid, block, 0, s, y, mean, rstd, x, w, b, M, C);
  else launch_k(k_layernorm_fwd<T, 8>, grid, block, 0, s, y, mean, rstd, x, w, b, M, C);
}

// ------------------------------------------------------------------ fixed-order partial sums
// out_j[c] = sum over parts of partials[p][j * seg + c] for j = 0..2: each
// block owns 32 columns with 32 warps; warp w sums parts w, w+32, ... in four
// interleaved accumulators (p = w + 32(4i + k) goes to accumulator k), combined
// as (a0 + a1) + (a2 + a3); the 32 warp sums are then added in warp order.
// Deterministic.
template <typename T>
__global__ void __launch_bounds__(1024)
    k_reduce_parts(T* __restrict__ o0, T* __restrict__ o1, T* __restrict__ o2,
                   const float* __restrict__ partials, int nparts, int width, int seg) {
  pdl_begin();
  __shared__ float sh[32][33];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * 32 + lane;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  if (c < width) {
    int p = warp;
    for (; p + 96 < nparts; p += 128) {
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[k] += partials[(long long)(p + 32 * k) * width + c];
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (p + 32 * k < nparts) acc[k] += partials[(long long)(p + 32 * k) * width + c];
  }
  sh[warp][lane] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
  __syncthreads();
  if (warp == 0 && c < width) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < 32; ++w) t += sh[w][lane];
    const int j = c / seg, cc = c % seg;
    T* o = j == 0 ? o0 : (j == 1 ? o1 : o2);
    if (o) o[cc] = from_f<T>(t);
  }
}

template <typename T>
static void reduce_parts(T* o0, T* o1, T* o2, const float* partials, int nparts, int width, int seg,
                         cudaStream_t s) {
  launch_k(k_reduce_parts<T>, (width + 31) / 32, 1024, 0, s, o0, o1, o2, partials, nparts, width, seg);
}

// ------------------------------------------------------------------ LayerNorm backward
// dx = rstd * (g - mean(g) - xhat * mean(g * xhat)),  g = dy * w.
// dres = (accumulate ? dres : 0) + dx in fp32; dres_b (if given) = storage copy.
// One warp per row.  All three row inputs (dy, x and the fp32 dres being
// accumulated into) are loaded together before the row reductions, so a warp
// keeps 6 KB (C = 768, bf16) in flight.  Column sums per block, each warp in
// its own shared-memory slice (no atomics): dw = sum dy * xhat, db = sum dy and,
// when dsum is wanted, the column sum of the new dres (the next projection's
// bias gradient).  A slice stores element (vector vi, lane e) at
// ((e / 4) * nv + vi) * 4 + e % 4, so a warp's float4 updates are conflict-free.
constexpr int kLnbBlocks = 592;
constexpr int kLnbWarps = 4;

__device__ __forceinline__ int lnb_slot(int vi, int e, int nv) { return (((e >> 2) * nv + vi) << 2) + (e & 3); }

template <typename T, int MAXV>
__global__ void __launch_bounds__(kLnbWarps * 32)
    k_layernorm_bwd(float* __restrict__ dres, T* __restrict__ dres_b, const T* __restrict__ dy,
                    const T* __restrict__ x, const float* __restrict__ mean,
                    const float* __restrict__ rstd, const T* __restrict__ w,
                    float* __restrict__ partials, int M, int C, int accumulate, int want_sum,
                    int rows_per_block) {
  pdl_begin();
  constexpr int N = V16<T>::N;
  extern __shared__ float sacc[];  // [kLnbWarps][3][C]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nv = C / N;
  float* mine = sacc + warp * 3 * C;
  for (int i = lane; i < 3 * C; i += 32) mine[i] = 0.f;
  __syncwarp();
  float wv[MAXV][N];
#pragma unroll
  for (int j = 0; j < MAXV; ++j) {
    int vi = lane + j * 32;
    if (vi < nv) load16(w + vi * N, wv[j]);
  }
  const int r0 = blockIdx.x * rows_per_block;
  const int r1 = min(M, r0 + rows_per_block);
  for (int r = r0 + warp; r < r1; r += kLnbWarps) {
    const float mu = mean[r], rs = rstd[r];
    float dyv[MAXV][N], xh[MAXV][N], d[MAXV][N];
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
      int vi = lane + j * 32;
      if (vi < nv) {
        load16(dy + (long long)r * C + vi * N, dyv[j]);
        load16(x + (long long)r * C + vi * N, xh[j]);
        if (accumulate) {
          const float* dp = dres + (long long)r * C + vi * N;
#pragma unroll
          for (int e = 0; e < N; e += 4) {
            float4 o = *reinterpret_cast<const float4*>(dp + e);
            d[j][e] = o.x; d[j][e + 1] = o.y; d[j][e + 2] = o.z; d[j][e + 3] = o.w;
          }
        } else {
#pragma unroll
          for (int e = 0; e < N; ++e) d[j][e] = 0.f;
        }
      }
    }
    float sg = 0.f, sgx = 0.f;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
      int vi = lane + j * 32;
      if (vi < nv) {
#pragma unroll
        for (int e = 0; e < N; ++e) {
          xh[j][e] = (xh[j][e] - mu) * rs;
          const float g = dyv[j][e] * wv[j][e];
          sg += g;
          sgx += g * xh[j][e];
        }
      }
    }
    sg = warp_sum(sg) / (float)C;
    sgx = warp_sum(sgx) / (float)C;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
      int vi = lane + j * 32;
      if (vi < nv) {
#pragma unroll
        for (int e = 0; e < N; ++e) d[j][e] += rs * (dyv[j][e] * wv[j][e] - sg - xh[j][e] * sgx);
        float* dp = dres + (long long)r * C + vi * N;
#pragma unroll
        for (int e = 0; e < N; e += 4)
          *reinterpret_cast<float4*>(dp + e) = make_float4(d[j][e], d[j][e + 1], d[j][e + 2], d[j][e + 3]);
        if (dres_b) store16(dres_b + (long long)r * C + vi * N, d[j]);
#pragma unroll
        for (int e = 0; e < N; e += 4) {
          float4* a0 = reinterpret_cast<float4*>(mine + lnb_slot(vi, e, nv));
          float4* a1 = reinterpret_cast<float4*>(mine + C + lnb_slot(vi, e, nv));
          float4 u = *a0, b = *a1;
          u.x += dyv[j][e] * xh[j][e]; u.y += dyv[j][e + 1] * xh[j][e + 1];
          u.z += dyv[j][e + 2] * xh[j][e + 2]; u.w += dyv[j][e + 3] * xh[j][e + 3];
          b.x += dyv[j][e]; b.y += dyv[j][e + 1]; b.z += dyv[j][e + 2]; b.w += dyv[j][e + 3];
          *a0 = u;
          *a1 = b;
          if (want_sum) {
            float4* a2 = reinterpret_cast<float4*>(mine + 2 * C + lnb_slot(vi, e, nv));
            float4 q = *a2;
            q.x += d[j][e]; q.y += d[j][e + 1]; q.z += d[j][e + 2]; q.w += d[j][e + 3];
            *a2 = q;
          }
        }
      }
    }
  }
  __syncthreads();
  const int width = (want_sum ? 3 : 2) * C;
  for (int i = threadIdx.x; i < width; i += blockDim.x) {
    const int kind = i / C, c = i - kind * C;
    const int slot = kind * C + lnb_slot(c / N, c % N, nv);
    float t = 0.f;
#pragma unroll
    for (int ww = 0; ww < kLnbWarps; ++ww) t += sacc[ww * 3 * C + slot];
    partials[(long long)blockIdx.x * width + i] = t;
  }
}

// Streaming variant for bf16 storage (C <= 2048): one persistent block of 8
// warps per SM.  Warp w of block b takes rows b*8 + w, + 8*gridDim.x, ...; lane
// 0 keeps the warp's next rows in flight with bulk copies (cp.async.bulk, one
// mbarrier per stage) into a ring of nbuf row stages [dy | x | dres] in shared
// memory, so a warp's memory stays busy while it computes.  Each row is read
// twice from shared memory (row sums, then the update).  The column sums for
// dw, db and dsum live in registers across all of the warp's rows; at the end
// the 8 warps add theirs in warp order and the block writes one partial row
// (the same fixed-order reduction follows).
constexpr int kLnsWarps = 8;
constexpr int kLnsBarBytes = 1024;

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ bool lns_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Warp-collective bounded wait (about 2 s of %globaltimer): lane 0 spins, every
// lane then observes the completed phase itself.
__device__ __forceinline__ bool lns_wait(uint32_t bar, uint32_t parity, int lane) {
  int ok = 1;
  if (lane == 0 && !lns_try_wait(bar, parity)) {
    const uint64_t t0 = globaltimer_ns();
    while (!lns_try_wait(bar, parity))
      if (globaltimer_ns() - t0 > 2000000000ull) { ok = 0; break; }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) (void)lns_try_wait(bar, parity);
  return ok != 0;
}
__device__ __forceinline__ void bf16x8_to_f(const uint4& q, float* v) {
  const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(u[i] << 16);
    v[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

template <int MAXV>
__global__ void __launch_bounds__(kLnsWarps * 32, 1)
    k_layernorm_bwd_stream(float* __restrict__ dres, bf16* __restrict__ dres_b, const bf16* __restrict__ dy,
                           const bf16* __restrict__ x, const float* __restrict__ mean,
                           const float* __restrict__ rstd, const bf16* __restrict__ w,
                           float* __restrict__ partials, int M, int C, int accumulate, int want_sum, int nbuf,
                           unsigned* status, int poison) {
  pdl_begin();
  extern __shared__ __align__(128) uint8_t lsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nv = C / 8;
  const uint32_t SB = 8u * (uint32_t)C;  // one row stage: dy, x (bf16), dres (fp32)
  uint8_t* mine = lsm + kLnsBarBytes + (size_t)warp * nbuf * SB;
  const uint32_t bar0 = smem_u32(lsm) + 8u * warp * nbuf;
  if (lane == 0) {
    for (int i = 0; i < nbuf; ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar0 + 8u * i) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  float wv[MAXV][8];
#pragma unroll
  for (int j = 0; j < MAXV; ++j) {
    const int vi = lane + j * 32;
    if (vi < nv) bf16x8_to_f(*reinterpret_cast<const uint4*>(w + vi * 8), wv[j]);
  }
  const int gw = blockIdx.x * kLnsWarps + warp, nw = gridDim.x * kLnsWarps;
  const int nrows = gw < M ? (M - 1 - gw) / nw + 1 : 0;
  const uint32_t tx = (accumulate ? 8u : 4u) * (uint32_t)C;
  auto issue = [&](int k) {  // lane 0: row k of this warp into stage k % nbuf
    if (poison && k == 0 && gw == 0) return;  // test hook: this row's copy never arrives
    const long long r = gw + (long long)k * nw;
    const int st = k % nbuf;
    const uint32_t dst = smem_u32(mine + (size_t)st * SB), bar = bar0 + 8u * st;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tx) : "memory");
    bulk_g2s(dst, dy + r * C, 2u * C, bar);
    bulk_g2s(dst + 2u * C, x + r * C, 2u * C, bar);
    if (accumulate) bulk_g2s(dst + 4u * C, dres + r * C, 4u * C, bar);
  };
  int issued = 0;
  if (lane == 0)
    for (; issued < nbuf - 1 && issued < nrows; ++issued) issue(issued);
  issued = __shfl_sync(0xffffffffu, issued, 0);
  float aw[MAXV][8], ab[MAXV][8], as[MAXV][8];
#pragma unroll
  for (int j = 0; j < MAXV; ++j)
#pragma unroll
    for (int e = 0; e < 8; ++e) aw[j][e] = ab[j][e] = as[j][e] = 0.f;
  const float invC = 1.0f / (float)C;
  float mu_n = 0.f, rs_n = 0.f;
  if (nrows > 0) { mu_n = mean[gw]; rs_n = rstd[gw]; }
  bool ok = true;
  int k = 0;
  for (; k < nrows; ++k) {
    if (issued < nrows) {  // refill the stage that row k - 1 used
      if (lane == 0) issue(issued);
      ++issued;
    }
    const long long r = gw + (long long)k * nw;
    const float mu = mu_n, rs = rs_n;
    if (k + 1 < nrows) { mu_n = mean[r + nw]; rs_n = rstd[r + nw]; }
    const int st = k % nbuf;
    if (!lns_wait(bar0 + 8u * st, (uint32_t)((k / nbuf) & 1), lane)) { ok = false; break; }
    const uint8_t* sp = mine + (size_t)st * SB;
    const bf16* sdy = reinterpret_cast<const bf16*>(sp);
    const bf16* sx = sdy + C;
    const float* sd = reinterpret_cast<const float*>(sp + 4u * C);
    float sg = 0.f, sgx = 0.f;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
      const int vi = lane + j * 32;
      if (vi < nv) {
        float a[8], b[8];
        bf16x8_to_f(*reinterpret_cast<const uint4*>(sdy + vi * 8), a);
        bf16x8_to_f(*reinterpret_cast<const uint4*>(sx + vi * 8), b);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float g = a[e] * wv[j][e];
          sg += g;
          sgx += g * ((b[e] - mu) * rs);
        }
      }
    }
    sg = warp_sum(sg) * invC;
    sgx = warp_sum(sgx) * invC;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
      const int vi = lane + j * 32;
      if (vi < nv) {
        float a[8], b[8], d[8];
        bf16x8_to_f(*reinterpret_cast<const uint4*>(sdy + vi * 8), a);
        bf16x8_to_f(*reinterpret_cast<const uint4*>(sx + vi * 8), b);
        if (accumulate) {
          const float4 d0 = *reinterpret_cast<const float4*>(sd + vi * 8);
          const float4 d1 = *reinterpret_cast<const float4*>(sd + vi * 8 + 4);
          d[0] = d0.x; d[1] = d0.y; d[2] = d0.z; d[3] = d0.w;
          d[4] = d1.x; d[5] = d1.y; d[6] = d1.z; d[7] = d1.w;
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) d[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float xh = (b[e] - mu) * rs;
          d[e] += rs * (a[e] * wv[j][e] - sg - xh * sgx);
          aw[j][e] += a[e] * xh;
          ab[j][e] += a[e];
          as[j][e] += d[e];
        }
        float* dp = dres + r * C + vi * 8;
        *reinterpret_cast<float4*>(dp) = make_float4(d[0], d[1], d[2], d[3]);
        *reinterpret_cast<float4*>(dp + 4) = make_float4(d[4], d[5], d[6], d[7]);
        if (dres_b) store16(dres_b + r * C + vi * 8, d);
      }
    }
    __syncwarp();  // every lane is done with this stage before lane 0 refills it
  }
  if (!ok) {
    if (status && lane == 0) atomicOr(status, ST_TIMEOUT);
    // never leave with bulk copies still landing in this warp's stages
    for (int kk = k; kk < issued; ++kk) (void)lns_wait(bar0 + 8u * (kk % nbuf), (uint32_t)((kk / nbuf) & 1), lane);
  }
  __syncthreads();
  // block partial: the 8 warps' column sums added in warp order
  float* red = reinterpret_cast<float*>(lsm + kLnsBarBytes);  // [warps][3][C]
  float* my = red + (size_t)warp * 3 * C;
#pragma unroll
  for (int j = 0; j < MAXV; ++j) {
    const int vi = lane + j * 32;
    if (vi < nv) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        my[vi * 8 + e] = aw[j][e];
        my[C + vi * 8 + e] = ab[j][e];
        my[2 * C + vi * 8 + e] = as[j][e];
      }
    }
  }
  __syncthreads();
  const int width = (want_sum ? 3 : 2) * C;
  for (int i = threadIdx.x; i < width; i += blockDim.x) {
    float t = 0.f;
#pragma unroll
    for (int ww = 0; ww < kLnsWarps; ++ww) t += red[(size_t)ww * 3 * C + i];
    partials[(long long)blockIdx.x * width + i] = t;
  }
}

size_t layernorm_bwd_partials_floats(int C) { return (size_t)kLnbBlocks * 3 * C; }

template <typename T>
void layernorm_bwd(float* dres, T* dres_b, const T* dy, const T* x, const float* mean,
                   const float* rstd, const T* w, T* dw, T* db, T* dsum, float* partials, int M,
                   int C, int accumulate, cudaStream_t s, unsigned* status) {
  if constexpr (sizeof(T) == 2) {
    // streaming kernel when at least two row stages per warp fit in shared memory
    const size_t budget = 227 * 1024 - kLnsBarBytes;
    int nbuf = (int)(budget / ((size_t)kLnsWarps * 8 * C));
    if (nbuf > 4) nbuf = 4;
    const int nv = C / 8, per = (nv + 31) / 32;
    if (nbuf >= 2 && per <= 8 && C % 8 == 0) {
      int nblocks = num_sms();
      const int want_rows = (M + kLnsWarps - 1) / kLnsWarps;
      if (nblocks > want_rows) nblocks = want_rows;
      if (nblocks > kLnbBlocks) nblocks = kLnbBlocks;
      const size_t sm = kLnsBarBytes + (size_t)kLnsWarps * nbuf * 8 * C;
      const int want_sum = dsum != nullptr;
#define LNS(P)                                                                                         \
  do {                                                                                                 \
    cudaFuncSetAttribute(k_layernorm_bwd_stream<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm); \
    launch_k(k_layernorm_bwd_stream<P>, nblocks, kLnsWarps * 32, sm, s, dres, (bf16*)dres_b, (const bf16*)dy, \
             (const bf16*)x, mean, rstd, (const bf16*)w, partials, M, C, accumulate, want_sum, nbuf, status, \
             (test_poison() & POISON_LN_BWD) ? 1 : 0);                                                 \
  } while (0)
      if (per <= 1) LNS(1);
      else if (per <= 2) LNS(2);
      else if (per <= 3) LNS(3);
      else if (per <= 4) LNS(4);
      else LNS(8);
#undef LNS
      reduce_parts<T>(dw, db, dsum, partials, nblocks, (want_sum ? 3 : 2) * C, C, s);
      return;
    }
  }
  const int nv = C / V16<T>::N;
  const int per = (nv + 31) / 32;
  int nblocks = (M + kLnbWarps - 1) / kLnbWarps;
  if (nblocks > kLnbBlocks) nblocks = kLnbBlocks;
  const int rpb = (M + nblocks - 1) / nblocks;
  const size_t sm = (size_t)kLnbWarps * 3 * C * sizeof(float);
  const int want_sum = dsum != nullptr;
#define LNB(P)                                                                                    \
  do {                                                                                            \
    if (sm > 48 * 1024)                                                                           \
      cudaFuncSetAttribute(k_layernorm_bwd<T, P>, cudaFuncAttributeMaxDynamicSharedMemorySize,    \
                           (int)sm);                                                              \
    launch_k(k_layernorm_bwd<T, P>, nblocks, kLnbWarps * 32, sm, s, dres, dres_b, dy, x, mean, rstd, w, \
                                                              partials, M, C, accumulate,         \
                                                              want_sum, rpb);                     \
  } while (0)
  if (per <= 1) LNB(1);
  else if (per <= 2) LNB(2);
  else if (per <= 3) LNB(3);
  else if (per <= 4) LNB(4);
  else LNB(8);
#undef LNB
  reduce_parts<T>(dw, db, dsum, partials, nblocks, (want_sum ? 3 : 2) * C, C, s);
}

// ------------------------------------------------------------------ column sums (bias grads)
constexpr int kColsumRowBlocks = 128;

template <typename T>
__global__ void __launch_bounds__(256)
    k_colsum_partial(float* __restrict__ partials, const T* __restrict__ x, int M, int N,
                     long long ld, int rows_per_block) {
  pdl_begin();
  constexpr int NV = V16<T>::N;
  __shared__ float sred[8][32 * NV];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = (blockIdx.x * 32 + lane) * NV;
  float acc[NV];
#pragma unroll
  for (int e = 0; e < NV; ++e) acc[e] = 0.f;
  const int r0 = blockIdx.y * rows_per_block, r1 = min(M, r0 + rows_per_block);
  if (c < N) {
    int r = r0 + warp;
    for (; r + 24 < r1; r += 32) {  // four rows in flight per warp
      uint4 q[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) q[k] = *reinterpret_cast<const uint4*>(x + (long long)(r + 8 * k) * ld + c);
      float v[4][NV];
#pragma unroll
      for (int k = 0; k < 4; ++k) unpack16<T>(q[k], v[k]);
#pragma unroll
      for (int e = 0; e < NV; ++e) acc[e] += (v[0][e] + v[1][e]) + (v[2][e] + v[3][e]);
    }
    for (; r < r1; r += 8) {
      float v[NV];
      load16(x + (long long)r * ld + c, v);
#pragma unroll
      for (int e = 0; e < NV; ++e) acc[e] += v[e];
    }
  }
#pragma unroll
  for (int e = 0; e < NV; ++e) sred[warp][lane * NV + e] = acc[e];
  __syncthreads();
  for (int i = threadIdx.x; i < 32 * NV; i += 256) {
    int cc = blockIdx.x * 32 * NV + i;
    float t = 0.f;
#pragma unroll
    for (int ww = 0; ww < 8; ++ww) t += sred[ww][i];
    if (cc < N) partials[(long long)blockIdx.y * N + cc] = t;
  }
}

size_t colsum_partials_floats(int N) { return (size_t)kColsumRowBlocks * N; }

template <typename T>
void colsum_reduce(T* out, const float* partials, int nparts, int N, cudaStream_t s) {
  reduce_parts<T>(out, (T*)nullptr, (T*)nullptr, partials, nparts, N, N, s);
}

template <typename T>
void colsum(T* out, const T* x, int M, int N, long long ld, float* partials, cudaStream_t s) {
  constexpr int NV = V16<T>::N;
  int nrb = (M + 127) / 128;
  if (nrb > kColsumRowBlocks) nrb = kColsumRowBlocks;
  const int rpb = (M + nrb - 1) / nrb;
  dim3 grid((N + 32 * NV - 1) / (32 * NV), nrb);
  launch_k(k_colsum_partial<T>, grid, 256, 0, s, partials, x, M, N, ld, rpb);
  reduce_parts<T>(out, (T*)nullptr, (T*)nullptr, partials, nrb, N, N, s);
}

// ------------------------------------------------------------------ elementwise
// gelu recompute for activation recompute: bf16 pairs through the same packed
// hardware-tanh arithmetic as the GEMM epilogue that produced them in the
// forward pass; fp32 through gelu_f, as the fp32 GEMM epilogue.  16-byte vectors.
template <typename T>
__global__ void __launch_bounds__(256) k_gelu_recompute(T* __restrict__ y, const T* __restrict__ x, long long n) {
  pdl_begin();
  constexpr int N = V16<T>::N;
  for (long long i = (blockIdx.x * (long long)blockDim.x + threadIdx.x) * N; i < n;
       i += (long long)gridDim.x * blockDim.x * N) {
    if constexpr (sizeof(T) == 2) {
      const uint4 u = ldg_stream(x + i);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float2 g, dg;
        gelu_and_grad2(make_float2(__uint_as_float(w[q] << 16), __uint_as_float(w[q] & 0xFFFF0000u)), g, dg);
        __nv_bfloat162 t = __floats2bfloat162_rn(g.x, g.y);
        o[q] = *reinterpret_cast<uint32_t*>(&t);
      }
      *reinterpret_cast<uint4*>(y + i) = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
      float v[N];
      load16(x + i, v);
#pragma unroll
      for (int e = 0; e < N; ++e) v[e] = gelu_f(v[e]);
      store16(y + i, v);
    }
  }
}
template <typename T> void gelu_recompute(T* y, const T* x, long long n, cudaStream_t s) {
  launch_k(k_gelu_recompute<T>, grid_for(n / V16<T>::N, 256, 148 * 8), 256, 0, s, y, x, n);
}

template <typename T>
__global__ void k_to_storage(T* __restrict__ dst, const float* __restrict__ src, long long n) {
  pdl_begin();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] = from_f<T>(src[i]);
}
template <typename T>
__global__ void k_to_f32(float* __restrict__ dst, const T* __restrict__ src, long long n) {
  pdl_begin();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] = to_f(src[i]);
}

template <typename T> void to_storage(T* dst, const float* src, long long n, cudaStream_t s) {
  launch_k(k_to_storage<T>, grid_for(n, 256), 256, 0, s, dst, src, n);
}
template <typename T> void to_f32(float* dst, const T* src, long long n, cudaStream_t s) {
  launch_k(k_to_f32<T>, grid_for(n, 256), 256, 0, s, dst, src, n);
}

// ------------------------------------------------------------------ cross-entropy
__device__ __forceinline__ float block_reduce(float v, float* sh, bool is_max) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = is_max ? warp_max(v) : warp_sum(v);
  __syncthreads();
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  float r = (lane < nw) ? sh[lane] : (is_max ? -INFINITY : 0.f);
  r = is_max ? warp_max(r) : warp_sum(r);
  return r;
}

// One block per row: lse = log sum_{n<V} exp z[n]; loss_row = lse - z[target].
template <typename T>
__global__ void k_ce_rowstats(const T* __restrict__ z, long long ldz, const int32_t* __restrict__ tgt,
                              int V, float* __restrict__ lse, float* __restrict__ loss_rows) {
  pdl_begin();
  __shared__ float sh[32];
  const int r = blockIdx.x;
  const T* zr = z + (long long)r * ldz;
  float m = -INFINITY;
  for (int c = threadIdx.x; c < V; c += blockDim.x) m = fmaxf(m, to_f(zr[c]));
  m = block_reduce(m, sh, true);
  float s = 0.f;
  for (int c = threadIdx.x; c < V; c += blockDim.x) s += expf(to_f(zr[c]) - m);
  s = block_reduce(s, sh, false);
  if (threadIdx.x == 0) {
    int t = tgt[r];
    t = (t < 0 || t >= V) ? 0 : t;
    float l = m + logf(s);
    lse[r] = l;
    loss_rows[r] = l - to_f(zr[t]);
  }
}
template <typename T>
void ce_rowstats(const T* z, long long ldz, const int32_t* tgt, int M, int V, float* lse,
                 float* loss_rows, cudaStream_t s) {
  launch_k(k_ce_rowstats<T>, M, 256, 0, s, z, ldz, tgt, V, lse, loss_rows);
}

// One warp per row: combine per-tile (max, sum exp) partials into lse.
__global__ void k_ce_reduce_partials(const float* __restrict__ pmax, const float* __restrict__ psum,
                                     int ntiles, int ld, const float* __restrict__ ztgt, int M,
                                     float* __restrict__ lse, float* __restrict__ loss_rows) {
  pdl_begin();
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (row >= M) return;
  const float* pm = pmax + (long long)row * ld;
  const float* ps = psum + (long long)row * ld;
  float m = -INFINITY;
  for (int i = lane; i < ntiles; i += 32) m = fmaxf(m, pm[i]);
  m = warp_max(m);
  float s = 0.f;
  for (int i = lane; i < ntiles; i += 32) {
    float mi = pm[i];
    if (mi > -INFINITY) s += ps[i] * expf(mi - m);
  }
  s = warp_sum(s);
  if (lane == 0) {
    float l = m + logf(s);
    lse[row] = l;
    loss_rows[row] = l - ztgt[row];
  }
}
void ce_reduce_partials(const float* pmax, const float* psum, int ntiles, int ld, const float* ztgt,
                        int M, float* lse, float* loss_rows, cudaStream_t s) {
  launch_k(k_ce_reduce_partials, (M * 32 + 255) / 256, 256, 0, s, pmax, psum, ntiles, ld, ztgt, M, lse,
                                                           loss_rows);
}

// dz = (softmax(z) - onehot(target)) * inv_scale on n < V, 0 on the pad columns; in place.
// e^(z - lse) is formed as 2^(z log2 e - lse log2 e) (one fma, one ex2.approx:
// relative error about 2^-22, far below the bf16 rounding of dz); each thread
// keeps two 16-byte vectors in flight.
template <typename T>
__global__ void __launch_bounds__(256)
    k_ce_dlogits(T* __restrict__ z, long long ldz, const float* __restrict__ lse,
                 const int32_t* __restrict__ tgt, int V, int Vpad, float inv_scale) {
  pdl_begin();
  constexpr int N = V16<T>::N;
  constexpr float L2E = 1.4426950408889634f;
  const int r = blockIdx.x;
  T* zr = z + (long long)r * ldz;
  const float nl = -lse[r] * L2E;
  int t = tgt[r];
  t = (t < 0 || t >= V) ? 0 : t;
  const int step = blockDim.x * N;
  auto dz = [&](int c0, float* v) {
#pragma unroll
    for (int e = 0; e < N; ++e) {
      const int c = c0 + e;
      float p = 0.f;
      if (c < V) asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(p) : "f"(fmaf(v[e], L2E, nl)));
      if (c == t) p -= 1.0f;
      v[e] = p * inv_scale;
    }
  };
  for (int c0 = threadIdx.x * N; c0 < Vpad; c0 += 2 * step) {
    const int c1 = c0 + step;
    float v0[N], v1[N];
    load16(zr + c0, v0);
    if (c1 < Vpad) load16(zr + c1, v1);
    dz(c0, v0);
    store16(zr + c0, v0);
    if (c1 < Vpad) {
      dz(c1, v1);
      store16(zr + c1, v1);
    }
  }
}
template <typename T>
void ce_dlogits(T* z, long long ldz, const float* lse, const int32_t* tgt, int M, int V, int Vpad,
                float inv_scale, cudaStream_t s) {
  launch_k(k_ce_dlogits<T>, M, 256, 0, s, z, ldz, lse, tgt, V, Vpad, inv_scale);
}

// Mean of M per-row values in a fixed order; flags a non-finite result.
__global__ void k_mean_reduce(float* out, const float* __restrict__ rows, int M, unsigned* status) {
  pdl_begin();
  __shared__ double sh[32];
  double s = 0.0;
  for (int i = threadIdx.x; i < M; i += blockDim.x) s += (double)rows[i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) sh[warp] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += sh[w];
    float r = (float)(t / (double)M);
    out[0] = r;
    if (!isfinite(r) && status) atomicOr(status, ST_NONFINITE);
  }
}
void mean_reduce(float* out, const float* rows, int M, unsigned* status, cudaStream_t s) {
  launch_k(k_mean_reduce, 1, 1024, 0, s, out, rows, M, status);
}

// ------------------------------------------------------------------ encoder backward
// Single-block bitonic sort of (token, position) keys: order[] lists positions
// grouped by token, ascending position within a token.  Keys live in shared
// memory (8 bytes each, M <= 16384).
__global__ void __launch_bounds__(1024) k_sort_tokens(uint32_t* __restrict__ order,
                                                      const int32_t* __restrict__ tok, int M, int V,
                                                      int P) {
  pdl_begin();
  extern __shared__ unsigned long long keys[];
  for (int i = threadIdx.x; i < P; i += blockDim.x) {
    unsigned long long k = ~0ull;
    if (i < M) {
      int t = tok[i];
      t = (t < 0 || t >= V) ? 0 : t;
      k = ((unsigned long long)(unsigned)t << 32) | (unsigned)i;
    }
    keys[i] = k;
  }
  __syncthreads();
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < P; i += blockDim.x) {
        int ixj = i ^ j;
        if (ixj > i) {
          unsigned long long a = keys[i], b = keys[ixj];
          bool up = (i & k) == 0;
          if ((a > b) == up) {
            keys[i] = b;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < M; i += blockDim.x) {
    order[i] = (uint32_t)(keys[i] & 0xffffffffull);
    order[M + i] = (uint32_t)(keys[i] >> 32);  // sorted token ids
  }
}

// The same sort for M <= 16384 positions and V <= 2^18 ids on 32-bit keys
// (id << 14 | position), bitonic over 16384 keys held 16 per thread: stages
// with partners inside a thread run in registers, inside a warp by shuffles,
// and only the 15 stages whose partners sit in another warp go through shared
// memory.  Keys are unique, so the result equals the 64-bit sort above.
constexpr int kSortKeys = 16384, kSortPerThread = 16, kSortPosBits = 14;

__device__ __forceinline__ void cmp_swap(uint32_t& a, uint32_t& b, bool up) {
  const uint32_t lo = min(a, b), hi = max(a, b);
  a = up ? lo : hi;
  b = up ? hi : lo;
}

// One bitonic stage (merge size K, partner distance J) on this thread's keys.
template <int K, int J>
__device__ __forceinline__ void sort_stage(uint32_t (&key)[kSortPerThread], int t, uint32_t* sk) {
  if constexpr (J < kSortPerThread) {
    // partner in this thread: element t*16 + r pairs with t*16 + (r ^ J)
#pragma unroll
    for (int r = 0; r < kSortPerThread; ++r) {
      if ((r & J) == 0) {
        const bool up = (((t * kSortPerThread + r) & K) == 0);
        cmp_swap(key[r], key[r | J], up);
      }
    }
  } else {
    constexpr int TJ = J / kSortPerThread;  // partner thread t ^ TJ, same r
    const bool up = (((t * kSortPerThread) & K) == 0);
    const bool keep_min = ((t & TJ) == 0) == up;
    if constexpr (TJ < 32) {
#pragma unroll
      for (int r = 0; r < kSortPerThread; ++r) {
        const uint32_t o = __shfl_xor_sync(0xffffffffu, key[r], TJ);
        key[r] = keep_min ? min(key[r], o) : max(key[r], o);
      }
    } else {
#pragma unroll
      for (int r = 0; r < kSortPerThread; ++r) sk[r * 1024 + t] = key[r];
      __syncthreads();
#pragma unroll
      for (int r = 0; r < kSortPerThread; ++r) {
        const uint32_t o = sk[r * 1024 + (t ^ TJ)];
        key[r] = keep_min ? min(key[r], o) : max(key[r], o);
      }
      __syncthreads();
    }
  }
}
template <int K, int J>
__device__ __forceinline__ void sort_merge(uint32_t (&key)[kSortPerThread], int t, uint32_t* sk) {
  if constexpr (J > 0) {
    sort_stage<K, J>(key, t, sk);
    sort_merge<K, J / 2>(key, t, sk);
  }
}
template <int K>
__device__ __forceinline__ void sort_levels(uint32_t (&key)[kSortPerThread], int t, uint32_t* sk) {
  if constexpr (K <= kSortKeys) {
    sort_merge<K, K / 2>(key, t, sk);
    sort_levels<K * 2>(key, t, sk);
  }
}

__global__ void __launch_bounds__(1024) k_sort_tokens32(uint32_t* __restrict__ order,
                                                        const int32_t* __restrict__ tok, int M, int V) {
  pdl_begin();
  extern __shared__ uint32_t sk32[];
  const int t = threadIdx.x;
  uint32_t key[kSortPerThread];
#pragma unroll
  for (int r = 0; r < kSortPerThread; ++r) {
    const int i = t * kSortPerThread + r;
    uint32_t k = 0xFFFFFFFFu;
    if (i < M) {
      int v = tok[i];
      v = (v < 0 || v >= V) ? 0 : v;
      k = ((uint32_t)v << kSortPosBits) | (uint32_t)i;
    }
    key[r] = k;
  }
  sort_levels<2>(key, t, sk32);
#pragma unroll
  for (int r = 0; r < kSortPerThread; ++r) {
    const int i = t * kSortPerThread + r;
    if (i < M) {
      order[i] = key[r] & ((1u << kSortPosBits) - 1u);
      order[M + i] = key[r] >> kSortPosBits;  // sorted token ids
    }
  }
}

void sort_tokens(uint32_t* order, const int32_t* tok, int M, int V, cudaStream_t s) {
  if (M <= kSortKeys && V <= (1 << (32 - kSortPosBits))) {
    const size_t sm = (size_t)kSortKeys * 4;
    cudaFuncSetAttribute(k_sort_tokens32, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    launch_k(k_sort_tokens32, 1, 1024, sm, s, order, tok, M, V);
    return;
  }
  int P = 1;
  while (P < M) P <<= 1;
  size_t sm = (size_t)P * 8;
  cudaFuncSetAttribute(k_sort_tokens, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  launch_k(k_sort_tokens, 1, 1024, sm, s, order, tok, M, V, P);
}

// Fixed summation order of the tied-embedding scatter: the positions holding
// token v, in ascending order, are cut into runs of kEncRun; each run is summed
// from zero in ascending order (fp32), the run sums are added in run order from
// zero, and dwte[v] = dwte[v] + total (one rounding to the storage type).  Runs
// spread the most frequent tokens over many blocks.
constexpr int kEncRun = 64;

// [s, e): the segment of the sorted token list holding stok[p] (stok ascending).
__device__ __forceinline__ void token_segment(const uint32_t* stok, int M, int p, int& s, int& e) {
  const uint32_t v = stok[p];
  int lo = 0, hi = p;  // first index with stok == v lies in [0, p]
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (stok[mid] < v) lo = mid + 1; else hi = mid;
  }
  s = lo;
  lo = p;
  hi = M;  // stok[lo] == v; find the first index > p with stok != v
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (stok[mid] == v) lo = mid; else hi = mid;
  }
  e = hi;
}

// One block per sorted index p; run heads sum their run.  A token with a single
// run finishes here (dwte update); otherwise the run sum is parked in the dx0 row
// of the run's first position, which no other run reads (dx0 is consumed).
template <typename T>
__global__ void __launch_bounds__(256)
    k_encoder_bwd_runs(T* __restrict__ dwte, float* __restrict__ dx0, const uint32_t* __restrict__ order,
                       int M, int C) {
  pdl_begin();
  const int p = blockIdx.x;
  const uint32_t* stok = order + M;
  int s, e;
  token_segment(stok, M, p, s, e);
  if ((p - s) % kEncRun) return;
  const int q = min(e, p + kEncRun);
  const bool single = e - s <= kEncRun;
  const uint32_t v = stok[p];
  for (int c = threadIdx.x * 4; c < C; c += blockDim.x * 4) {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    int r = p;
    for (; r + 8 <= q; r += 8) {
      float4 u[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) u[k] = *reinterpret_cast<const float4*>(dx0 + (long long)order[r + k] * C + c);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        a0 = a0 + u[k].x; a1 = a1 + u[k].y; a2 = a2 + u[k].z; a3 = a3 + u[k].w;
      }
    }
    for (; r < q; ++r) {
      float4 u = *reinterpret_cast<const float4*>(dx0 + (long long)order[r] * C + c);
      a0 = a0 + u.x; a1 = a1 + u.y; a2 = a2 + u.z; a3 = a3 + u.w;
    }
    if (single) {
      T* dst = dwte + (long long)v * C + c;
      dst[0] = from_f<T>(to_f(dst[0]) + a0);
      dst[1] = from_f<T>(to_f(dst[1]) + a1);
      dst[2] = from_f<T>(to_f(dst[2]) + a2);
      dst[3] = from_f<T>(to_f(dst[3]) + a3);
    } else {
      *reinterpret_cast<float4*>(dx0 + (long long)order[p] * C + c) = make_float4(a0, a1, a2, a3);
    }
  }
}

// One block per segment head of a token with more than one run: add the
// parked run sums in run order, then update dwte once.
template <typename T>
__global__ void __launch_bounds__(256)
    k_encoder_bwd_combine(T* __restrict__ dwte, const float* __restrict__ dx0,
                          const uint32_t* __restrict__ order, int M, int C) {
  pdl_begin();
  const int p = blockIdx.x;
  const uint32_t* stok = order + M;
  const uint32_t v = stok[p];
  if (p > 0 && stok[p - 1] == v) return;
  int s, e;
  token_segment(stok, M, p, s, e);
  if (e - s <= kEncRun) return;
  for (int c = threadIdx.x * 4; c < C; c += blockDim.x * 4) {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    for (int r = s; r < e; r += kEncRun) {
      const float4 u = *reinterpret_cast<const float4*>(dx0 + (long long)order[r] * C + c);
      a0 = a0 + u.x; a1 = a1 + u.y; a2 = a2 + u.z; a3 = a3 + u.w;
    }
    T* dst = dwte + (long long)v * C + c;
    dst[0] = from_f<T>(to_f(dst[0]) + a0);
    dst[1] = from_f<T>(to_f(dst[1]) + a1);
    dst[2] = from_f<T>(to_f(dst[2]) + a2);
    dst[3] = from_f<T>(to_f(dst[3]) + a3);
  }
}

// dwpe[t, c] = sum over b ascending of dx0[b, t, c] (fp32), stored once.
template <typename T>
__global__ void k_encoder_bwd_wpe(T* __restrict__ dwpe, const float* __restrict__ dx0, int B, int Tn,
                                  int C) {
  pdl_begin();
  long long n = (long long)Tn * C;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    float acc = 0.f;
    for (int b = 0; b < B; ++b) acc = acc + dx0[(long long)b * n + i];
    dwpe[i] = from_f<T>(acc);
  }
}

template <typename T>
void encoder_bwd(T* dwte, T* dwpe, float* dx0, const uint32_t* order, const int32_t* tok, int B,
                 int Tn, int C, cudaStream_t s) {
  const int M = B * Tn;
  int threads = C / 4;
  if (threads > 256) threads = 256;
  if (threads < 32) threads = 32;
  // dwpe first: the run kernel overwrites some dx0 rows with run sums
  launch_k(k_encoder_bwd_wpe<T>, grid_for((long long)Tn * C, 256), 256, 0, s, dwpe, dx0, B, Tn, C);
  launch_k(k_encoder_bwd_runs<T>, M, threads, 0, s, dwte, dx0, order, M, C);
  launch_k(k_encoder_bwd_combine<T>, M, threads, 0, s, dwte, dx0, order, M, C);
}

// ------------------------------------------------------------------ split-K reduction
// Rows blockIdx.y, + gridDim.y, ... of the output, a float4 of columns per
// thread; the splits are added in split order (four loads in flight at a time).
__global__ void k_splitk_reduce(void* __restrict__ out, int out_f32, long long ldo,
                                const float* __restrict__ ws, int splits, int M, int N) {
  pdl_begin();
  const int n = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (n >= N) return;
  const long long plane = (long long)M * N;
  for (int m = blockIdx.y; m < M; m += gridDim.y) {
    const float* src = ws + (long long)m * N + n;
    float4 a = *reinterpret_cast<const float4*>(src);
    int sp = 1;
    for (; sp + 3 < splits; sp += 4) {
      float4 b[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) b[k] = *reinterpret_cast<const float4*>(src + (sp + k) * plane);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        a.x += b[k].x; a.y += b[k].y; a.z += b[k].z; a.w += b[k].w;
      }
    }
    for (; sp < splits; ++sp) {
      const float4 b = *reinterpret_cast<const float4*>(src + sp * plane);
      a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
    }
    if (out_f32) {
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + (long long)m * ldo + n) = a;
    } else {
      bf16* o = reinterpret_cast<bf16*>(out) + (long long)m * ldo + n;
      __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y), hi = __floats2bfloat162_rn(a.z, a.w);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&lo);
      u.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(o) = u;
    }
  }
}
void splitk_reduce(void* out, int out_f32, long long ldo, const float* ws, int splits, int M, int N,
                   cudaStream_t s) {
  const dim3 grid((unsigned)((N / 4 + 255) / 256), (unsigned)(M < 65535 ? M : 65535));
  launch_k(k_splitk_reduce, grid, 256, 0, s, out, out_f32, ldo, ws, splits, M, N);
}

// ------------------------------------------------------------------ global norm + AdamW
// Sum of squares of n gradient values in nparts fixed slices (one partial per
// block, fixed order).  Each thread keeps four 16-byte loads in flight.
template <typename G>
__global__ void __launch_bounds__(512)
    k_sumsq(float* __restrict__ partials, const G* __restrict__ g, long long n, long long chunk) {
  pdl_begin();
  constexpr int N = V16<G>::N;
  __shared__ float sh[32];
  const long long b0 = blockIdx.x * chunk;
  const long long b1 = min(n, b0 + chunk);
  const long long step = (long long)blockDim.x * N;
  float s[4] = {0.f, 0.f, 0.f, 0.f};
  long long i = b0 + (long long)threadIdx.x * N;
  for (; i + 3 * step < b1; i += 4 * step) {
    float v[4][N];
#pragma unroll
    for (int u = 0; u < 4; ++u) load16(g + i + u * step, v[u]);
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int e = 0; e < N; ++e) s[u] = fmaf(v[u][e], v[u][e], s[u]);
  }
  for (; i < b1; i += step) {
    float v[N];
    load16(g + i, v);
#pragma unroll
    for (int e = 0; e < N; ++e) s[0] = fmaf(v[e], v[e], s[0]);
  }
  const float t = block_reduce((s[0] + s[1]) + (s[2] + s[3]), sh, false);
  if (threadIdx.x == 0) partials[blockIdx.x] = t;
}
template <typename G>
void grad_sumsq_partials(float* partials, int nparts, const G* g, long long n, cudaStream_t s) {
  constexpr int N = V16<G>::N;
  long long chunk = (n + nparts - 1) / nparts;
  chunk = (chunk + N - 1) / N * N;
  launch_k(k_sumsq<G>, nparts, 512, 0, s, partials, g, n, chunk);
}

// Norm, clip scale, bias corrections and the update guard (see GuardState).
// t = host_t when > 0, else the device step counter + 1 (stored unless the
// update is skipped).
__global__ void __launch_bounds__(1024)
    k_norm_finalize(float* norm_scale, const float* __restrict__ partials, int nparts, float max_norm,
                    unsigned* status, int* counter, int host_t, float b1, float b2,
                    const OptHyper* __restrict__ hp, const float* __restrict__ loss, GuardState* guard) {
  pdl_begin();
  if (hp) {
    max_norm = hp->max_norm;
    host_t = hp->t;
    b1 = hp->b1;
    b2 = hp->b2;
  }
  __shared__ double sh[5][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  // [0]: the squared-gradient partials; [1..4]: the guard's window sums of the held
  // losses, their squares, the held norms and their squares
  double q[5] = {0.0, 0.0, 0.0, 0.0, 0.0};
  for (int i = threadIdx.x; i < nparts; i += blockDim.x) q[0] += (double)partials[i];
  const int held = guard ? guard->count : 0;
  if (guard && threadIdx.x < held) {
    const double lv = guard->loss_hist[threadIdx.x], nv = guard->norm_hist[threadIdx.x];
    q[1] = lv; q[2] = lv * lv; q[3] = nv; q[4] = nv * nv;
  }
#pragma unroll
  for (int k = 0; k < 5; ++k)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) q[k] += __shfl_xor_sync(0xffffffffu, q[k], o);
  if (lane == 0)
#pragma unroll
    for (int k = 0; k < 5; ++k) sh[k][warp] = q[k];
  __syncthreads();
  if (threadIdx.x == 0) {
    double t[5] = {0.0, 0.0, 0.0, 0.0, 0.0};
    for (int w = 0; w < nwarps; ++w)
#pragma unroll
      for (int k = 0; k < 5; ++k) t[k] += sh[k][w];
    const float norm = (float)sqrt(t[0]);
    const float lv = loss ? *loss : 0.f;
    norm_scale[0] = norm;
    norm_scale[1] = (norm > max_norm) ? max_norm / norm : 1.0f;
    const bool finite = isfinite(norm) && isfinite(lv);
    if (!finite && status) atomicOr(status, ST_NONFINITE);
    bool skip = !finite;
    if (guard) {
      float zl = __int_as_float(0x7fc00000), zn = zl;  // NaN until the window is full
      if (held >= guard->window) {
        const double sl = t[1], sl2 = t[2], sn = t[3], sn2 = t[4];
        const double n = (double)held;
        const double ml = sl / n, mn = sn / n;
        const double vl = fmax(sl2 / n - ml * ml, 0.0), vn = fmax(sn2 / n - mn * mn, 0.0);
        zl = vl > 0.0 ? (float)(((double)lv - ml) / sqrt(vl)) : ((double)lv == ml ? 0.f : (float)copysign(INFINITY, (double)lv - ml));
        zn = vn > 0.0 ? (float)(((double)norm - mn) / sqrt(vn)) : ((double)norm == mn ? 0.f : (float)copysign(INFINITY, (double)norm - mn));
      }
      guard->z_loss = zl;
      guard->z_norm = zn;
      const bool spike = finite && ((guard->loss_z_max > 0.f && zl > guard->loss_z_max) ||
                                    (guard->norm_z_max > 0.f && zn > guard->norm_z_max));
      if (!finite) guard->skipped_nonfinite += 1;
      if (spike) guard->skipped_spike += 1;
      skip = skip || spike;
      guard->last_skipped = skip ? 1 : 0;
      if (finite) {  // every finite observation enters the window, skipped or not
        const int hd = guard->head;
        guard->loss_hist[hd] = lv;
        guard->norm_hist[hd] = norm;
        guard->head = hd + 1 == guard->window ? 0 : hd + 1;
        if (guard->count < guard->window) guard->count += 1;
      }
    }
    norm_scale[4] = skip ? 1.f : 0.f;
    const int step = host_t > 0 ? host_t : counter[0] + 1;
    if (!skip) counter[0] = step;
    norm_scale[2] = 1.0f - powf(b1, (float)step);
    norm_scale[3] = 1.0f - powf(b2, (float)step);
  }
}
void grad_norm_finalize(float* norm_scale, const float* partials, int nparts, float max_norm,
                        unsigned* status, int* counter, int host_t, float b1, float b2,
                        const OptHyper* hp, const float* loss, GuardState* guard, cudaStream_t s) {
  launch_k(k_norm_finalize, 1, 1024, 0, s, norm_scale, partials, nparts, max_norm, status, counter,
           host_t, b1, b2, hp, loss, guard);
}

struct SegTable { Segment s[kMaxSegments]; int n; };

template <typename G> struct G4;
template <> struct G4<float> {
  static __device__ __forceinline__ void ld(const float* p, float* o) {
    float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
  static __device__ __forceinline__ void st(float* p, const float* o) {
    *reinterpret_cast<float4*>(p) = make_float4(o[0], o[1], o[2], o[3]);
  }
};
template <> struct G4<bf16> {
  static __device__ __forceinline__ void ld(const bf16* p, float* o) {
    uint2 u = *reinterpret_cast<const uint2*>(p);
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&u.x), b = *reinterpret_cast<__nv_bfloat162*>(&u.y);
    o[0] = __low2float(a); o[1] = __high2float(a); o[2] = __low2float(b); o[3] = __high2float(b);
  }
  static __device__ __forceinline__ void st(bf16* p, const float* o) {
    __nv_bfloat162 a = __floats2bfloat162_rn(o[0], o[1]), b = __floats2bfloat162_rn(o[2], o[3]);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
  }
};

// acc = (first ? 0 : acc) + scale * g, four values per thread and step.
// The loss is accumulated the same way (acc_loss = (first ? 0 : acc_loss) + scale * loss),
// so the update guard sees the mean loss of the accumulated micro-batches.
template <typename G>
__global__ void __launch_bounds__(256)
    k_grad_acc(float* __restrict__ acc, const G* __restrict__ g, long long n, float scale, int first,
               const float* __restrict__ loss, float* __restrict__ acc_loss) {
  pdl_begin();
  if (blockIdx.x == 0 && threadIdx.x == 0 && loss) *acc_loss = fmaf(scale, *loss, first ? 0.f : *acc_loss);
  const long long n4 = n / 4;
  for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < n4;
       q += (long long)gridDim.x * blockDim.x) {
    const long long i = q * 4;
    float a[4] = {0.f, 0.f, 0.f, 0.f}, b[4];
    G4<G>::ld(g + i, b);
    if (!first) G4<float>::ld(acc + i, a);
#pragma unroll
    for (int e = 0; e < 4; ++e) a[e] = fmaf(scale, b[e], a[e]);
    G4<float>::st(acc + i, a);
  }
  if (blockIdx.x == 0 && threadIdx.x < (int)(n - n4 * 4)) {
    const long long i = n4 * 4 + threadIdx.x;
    acc[i] = fmaf(scale, to_f(g[i]), first ? 0.f : acc[i]);
  }
}
template <typename G>
void grad_accumulate(float* acc, const G* g, long long n, float scale, int first, const float* loss,
                     float* acc_loss, cudaStream_t s) {
  launch_k(k_grad_acc<G>, grid_for(n / 4 + 1, 256, 148 * 8), 256, 0, s, acc, g, n, scale, first, loss, acc_loss);
}
template void grad_accumulate<float>(float*, const float*, long long, float, int, const float*, float*,
                                     cudaStream_t);
template void grad_accumulate<bf16>(float*, const bf16*, long long, float, int, const float*, float*,
                                    cudaStream_t);

// m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2; w -= lr (m/bc1 / (sqrt(v/bc2) + eps) + wd_seg w)
// with g = grad * clip_scale; clip scale and bias corrections come from
// norm_scale[1..3] on the device; one pass over 4-element vectors.
template <typename G, typename P>
__global__ void __launch_bounds__(256)
    k_adamw(float* __restrict__ master, P* __restrict__ pcopy, const G* __restrict__ grad,
            float* __restrict__ m, float* __restrict__ v, long long n, SegTable segs,
            const float* __restrict__ norm_scale, float lr, float b1, float b2, float eps,
            float wd, const OptHyper* __restrict__ hp) {
  pdl_begin();
  if (hp) {
    lr = hp->lr;
    b1 = hp->b1;
    b2 = hp->b2;
    eps = hp->eps;
    wd = hp->wd;
  }
  if (norm_scale[4] != 0.f) return;  // the guard skipped this update: master, m, v stay as they are
  const float sc = norm_scale[1], bc1 = norm_scale[2], bc2 = norm_scale[3];
  const long long n4 = n / 4;
  // the segments tile [0, n) in ascending order and each thread's i only grows,
  // so its current segment is found by stepping forward from the last one
  int seg = 0;
  for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < n4;
       q += (long long)gridDim.x * blockDim.x) {
    const long long i = q * 4;
    while (seg < segs.n && i >= segs.s[seg].end) ++seg;
    const float lam = (seg < segs.n && i >= segs.s[seg].begin && segs.s[seg].decay) ? wd : 0.f;
    float w[4], g[4], mm[4], vv[4];
    G4<float>::ld(master + i, w);
    G4<G>::ld(grad + i, g);
    G4<float>::ld(m + i, mm);
    G4<float>::ld(v + i, vv);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float gg = g[e] * sc;
      mm[e] = b1 * mm[e] + (1.0f - b1) * gg;
      vv[e] = b2 * vv[e] + (1.0f - b2) * gg * gg;
      float mh = mm[e] / bc1, vh = vv[e] / bc2;
      w[e] = w[e] - lr * (mh / (sqrtf(vh) + eps) + lam * w[e]);
    }
    G4<float>::st(master + i, w);
    G4<float>::st(m + i, mm);
    G4<float>::st(v + i, vv);
    if (pcopy) G4<P>::st(pcopy + i, w);
  }
}

template <typename G, typename P>
void adamw(float* master, P* param_copy, const G* grad, float* m, float* v, long long n,
           const Segment* segs, int nsegs, const float* norm_scale, float lr, float beta1,
           float beta2, float eps, float wd, const OptHyper* hp, cudaStream_t s) {
  SegTable t;
  t.n = nsegs;
  for (int i = 0; i < nsegs && i < kMaxSegments; ++i) t.s[i] = segs[i];
  launch_k(k_adamw<G, P>, grid_for(n / 4, 256, 148 * 8), 256, 0, s, master, param_copy, grad, m, v, n, t,
           norm_scale, lr, beta1, beta2, eps, wd, hp);
}

// ------------------------------------------------------------------ instantiations
#define INST(T)                                                                                     \
  template void encoder_fwd<T>(T*, const int32_t*, const T*, const T*, int, int, int, int,         \
                               unsigned*, cudaStream_t);                                           \
  template void layernorm_fwd<T>(T*, float*, float*, const T*, const T*, const T*, int, int,       \
                                 cudaStream_t);                                                    \
  template void layernorm_bwd<T>(float*, T*, const T*, const T*, const float*, const float*,       \
                                 const T*, T*, T*, T*, float*, int, int, int, cudaStream_t,        \
                                 unsigned*);                                                        \
  template void colsum<T>(T*, const T*, int, int, long long, float*, cudaStream_t);                \
  template void colsum_reduce<T>(T*, const float*, int, int, cudaStream_t);                        \
  template void gelu_recompute<T>(T*, const T*, long long, cudaStream_t);                          \
  template void to_storage<T>(T*, const float*, long long, cudaStream_t);                          \
  template void to_f32<T>(float*, const T*, long long, cudaStream_t);                              \
  template void ce_rowstats<T>(const T*, long long, const int32_t*, int, int, float*, float*,      \
                               cudaStream_t);                                                      \
  template void ce_dlogits<T>(T*, long long, const float*, const int32_t*, int, int, int, float,   \
                              cudaStream_t);                                                       \
  template void encoder_bwd<T>(T*, T*, float*, const uint32_t*, const int32_t*, int, int,    \
                               int, cudaStream_t);                                                 \
  template void grad_sumsq_partials<T>(float*, int, const T*, long long, cudaStream_t);
INST(float)
INST(bf16)
#undef INST
template void adamw<float, float>(float*, float*, const float*, float*, float*, long long,
                                  const Segment*, int, const float*, float, float, float, float,
                                  float, const OptHyper*, cudaStream_t);
template void adamw<bf16, bf16>(float*, bf16*, const bf16*, float*, float*, long long,
                                const Segment*, int, const float*, float, float, float, float,
                                float, const OptHyper*, cudaStream_t);
template void adamw<float, bf16>(float*, bf16*, const float*, float*, float*, long long,
                                 const Segment*, int, const float*, float, float, float, float,
                                 float, const OptHyper*, cudaStream_t);

}  // namespace gpt2k
