// Causal multi-head attention, forward and backward, never materialising the
// T x T score matrix (online softmax over 64-key tiles, FlashAttention-style;
// "Let's reproduce GPT-2 (124M)" wiki page, "GPU optimisation ladder":
// FlashAttention gives the same result without storing T x T).
//
// bf16 path (d = 64): warp-level bf16 tensor-core MMA (m16n8k16, fp32
// accumulate), 64-query x 64-key tiles, cp.async double-buffered K/V tiles in
// XOR-swizzled shared memory, probabilities kept in registers.
// Backward is deterministic: one kernel owns each 64-row block of dK/dV and
// loops over query blocks, another owns each block of dQ and loops over key
// blocks (no float atomics).
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

#define LOG2E 1.4426950408889634f
#define LN2 0.6931471805599453f

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;"); }
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 64 x 64 bf16 tile, 8 chunks of 16 B per row, chunk index XOR (row & 7).
__device__ __forceinline__ uint32_t tile_off(int r, int chunk) {
  return (uint32_t)(r * 128 + ((chunk ^ (r & 7)) << 4));
}

// Async copy of rows [r0, r0+64) of a [T, 64] strided matrix into a swizzled tile.
__device__ __forceinline__ void load_tile(uint32_t sbase, const bf16* g, long long st, int r0, int T,
                                          int tid, int nthreads) {
  for (int i = tid; i < 512; i += nthreads) {
    int r = i >> 3, c = i & 7;
    int gr = r0 + r;
    bool ok = gr < T;
    const bf16* src = g + (long long)(ok ? gr : 0) * st + c * 8;
    cp_async16(sbase + tile_off(r, c), src, ok);
  }
}

// A-operand fragments (16 rows x 64 cols, 4 k-steps) of rows [row0, row0+16) of a tile.
__device__ __forceinline__ void load_afrag(uint32_t sbase, int row0, int lane, uint32_t (*f)[4]) {
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    int r = row0 + (lane & 7) + ((lane >> 3) & 1) * 8;
    int c = kk * 2 + (lane >> 4);
    ldsm_x4(sbase + tile_off(r, c), f[kk][0], f[kk][1], f[kk][2], f[kk][3]);
  }
}

// acc[8][4] (16 x 64) += A(16 x 64, regs) * tile^T, tile rows are the n index.
__device__ __forceinline__ void mma_a_tileT(float (*acc)[4], const uint32_t (*a)[4], uint32_t sbase,
                                            int lane) {
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      int r = np * 16 + (lane & 7) + ((lane >> 4) << 3);
      int c = kk * 2 + ((lane >> 3) & 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(sbase + tile_off(r, c), b0, b1, b2, b3);
      mma16816(acc[2 * np], a[kk], b0, b1);
      mma16816(acc[2 * np + 1], a[kk], b2, b3);
    }
  }
}

// acc[8][4] (16 x 64) += P(16 x 64 keys, from accumulator regs) * tile (64 keys x 64 cols).
__device__ __forceinline__ void mma_p_tile(float (*acc)[4], const float (*p)[4], uint32_t sbase,
                                           int lane) {
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    uint32_t a[4];
    a[0] = pack_bf16(p[2 * kk][0], p[2 * kk][1]);
    a[1] = pack_bf16(p[2 * kk][2], p[2 * kk][3]);
    a[2] = pack_bf16(p[2 * kk + 1][0], p[2 * kk + 1][1]);
    a[3] = pack_bf16(p[2 * kk + 1][2], p[2 * kk + 1][3]);
#pragma unroll
    for (int dp = 0; dp < 4; ++dp) {
      int r = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
      int c = dp * 2 + (lane >> 4);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(sbase + tile_off(r, c), b0, b1, b2, b3);
      mma16816(acc[2 * dp], a, b0, b1);
      mma16816(acc[2 * dp + 1], a, b2, b3);
    }
  }
}

__device__ __forceinline__ void zero_acc(float (*a)[4]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i][0] = a[i][1] = a[i][2] = a[i][3] = 0.f;
}

// ------------------------------------------------------------------ forward (bf16)
__global__ void __launch_bounds__(128) k_attn_fwd_bf16(AttnArgs a) {
  __shared__ __align__(128) uint8_t smem[8192 * 5];
  const uint32_t sQ = smem_u32(smem), sK0 = sQ + 8192, sV0 = sQ + 3 * 8192;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nqb = gridDim.x;
  const int qb = nqb - 1 - blockIdx.x;
  const int b = blockIdx.y / a.H, h = blockIdx.y % a.H;
  const int T = a.T;
  const bf16* Q = static_cast<const bf16*>(a.q) + b * a.sb + h * a.sh;
  const bf16* K = static_cast<const bf16*>(a.k) + b * a.sb + h * a.sh;
  const bf16* Vp = static_cast<const bf16*>(a.v) + b * a.sb + h * a.sh;
  const int q0 = qb * 64;
  load_tile(sQ, Q, a.st, q0, T, tid, 128);
  load_tile(sK0, K, a.st, 0, T, tid, 128);
  load_tile(sV0, Vp, a.st, 0, T, tid, 128);
  cp_commit();
  cp_wait_all();
  __syncthreads();
  uint32_t qf[4][4];
  load_afrag(sQ, warp * 16, lane, qf);
  float o[8][4];
  zero_acc(o);
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const float c2 = a.scale * LOG2E;
  const int g = lane >> 2, t4 = lane & 3;
  const int i0 = q0 + warp * 16 + g;  // query rows i0 and i0 + 8
  for (int kb = 0; kb <= qb; ++kb) {
    const int st = kb & 1;
    const uint32_t sK = sK0 + st * 8192, sV = sV0 + st * 8192;
    if (kb + 1 <= qb) {
      load_tile(sK0 + (st ^ 1) * 8192, K, a.st, (kb + 1) * 64, T, tid, 128);
      load_tile(sV0 + (st ^ 1) * 8192, Vp, a.st, (kb + 1) * 64, T, tid, 128);
      cp_commit();
    }
    float s[8][4];
    zero_acc(s);
    mma_a_tileT(s, qf, sK, lane);
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = kb * 64 + nt * 8 + 2 * t4 + (e & 1);
        const int i = i0 + ((e >> 1) << 3);
        float v = s[nt][e] * c2;
        if (kb == qb && j > i) v = -INFINITY;
        s[nt][e] = v;
        mx[e >> 1] = fmaxf(mx[e >> 1], v);
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    }
    float corr[2], mnew[2], rs[2] = {0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mnew[r] = fmaxf(mrow[r], mx[r]);
      corr[r] = exp2f(mrow[r] - mnew[r]);
      mrow[r] = mnew[r];
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float p = exp2f(s[nt][e] - mnew[e >> 1]);
        s[nt][e] = p;
        rs[e >> 1] += p;
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 1);
      rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 2);
      lrow[r] = lrow[r] * corr[r] + rs[r];
    }
#pragma unroll
    for (int dt = 0; dt < 8; ++dt) {
      o[dt][0] *= corr[0]; o[dt][1] *= corr[0];
      o[dt][2] *= corr[1]; o[dt][3] *= corr[1];
    }
    mma_p_tile(o, s, sV, lane);
    cp_wait_all();
    __syncthreads();
  }
  bf16* O = static_cast<bf16*>(a.o) + b * a.osb + h * a.osh;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int i = i0 + r * 8;
    if (i >= T) continue;
    const float inv = 1.0f / lrow[r];
#pragma unroll
    for (int dt = 0; dt < 8; ++dt) {
      uint32_t pk = pack_bf16(o[dt][2 * r] * inv, o[dt][2 * r + 1] * inv);
      *reinterpret_cast<uint32_t*>(O + (long long)i * a.ost + dt * 8 + 2 * t4) = pk;
    }
    if (t4 == 0) a.lse[((long long)blockIdx.y) * T + i] = (mrow[r] + log2f(lrow[r])) * LN2;
  }
}

// ------------------------------------------------------------------ backward (bf16)
// D[b, h, i] = sum_c dO[i, c] * O[i, c]   (one warp per row)
template <typename T>
__global__ void k_attn_rowdot(AttnArgs a) {
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

// dK, dV for a 64-key block: loop over query blocks qb >= kb.
__global__ void __launch_bounds__(128) k_attn_bwd_dkdv_bf16(AttnArgs a) {
  __shared__ __align__(128) uint8_t smem[8192 * 4];
  __shared__ float sL[2][64], sD[2][64];
  const uint32_t sQ0 = smem_u32(smem), sO0 = sQ0 + 2 * 8192;  // Q / dO double buffers
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = gridDim.x;
  const int kb = blockIdx.x;
  const int bh = blockIdx.y;
  const int b = bh / a.H, h = bh % a.H;
  const int T = a.T;
  const long long off = b * a.sb + h * a.sh, ooff = b * a.osb + h * a.osh;
  const bf16* Q = static_cast<const bf16*>(a.q) + off;
  const bf16* K = static_cast<const bf16*>(a.k) + off;
  const bf16* Vp = static_cast<const bf16*>(a.v) + off;
  const bf16* dO = static_cast<const bf16*>(a.dO) + ooff;
  const float* lse = a.lse + (long long)bh * T;
  const float* Dv = a.Dbuf + (long long)bh * T;
  const int k0 = kb * 64;
  // K and V tiles are parked in the stage-1 buffers until their fragments are in registers
  load_tile(sQ0 + 8192, K, a.st, k0, T, tid, 128);
  load_tile(sO0 + 8192, Vp, a.st, k0, T, tid, 128);
  load_tile(sQ0, Q, a.st, k0, T, tid, 128);
  load_tile(sO0, dO, a.ost, k0, T, tid, 128);
  cp_commit();
  if (tid < 64) {
    int i = k0 + tid;
    sL[0][tid] = (i < T) ? lse[i] * LOG2E : INFINITY;
    sD[0][tid] = (i < T) ? Dv[i] : 0.f;
  }
  cp_wait_all();
  __syncthreads();
  uint32_t kf[4][4], vf[4][4];
  load_afrag(sQ0 + 8192, warp * 16, lane, kf);
  load_afrag(sO0 + 8192, warp * 16, lane, vf);
  __syncthreads();
  float dk[8][4], dv[8][4];
  zero_acc(dk);
  zero_acc(dv);
  const float c2 = a.scale * LOG2E;
  const int g = lane >> 2, t4 = lane & 3;
  const int j0 = k0 + warp * 16 + g;  // key rows j0, j0 + 8
  for (int qb = kb; qb < nb; ++qb) {
    const int st = (qb - kb) & 1;
    const uint32_t sQ = sQ0 + st * 8192, sO = sO0 + st * 8192;
    if (qb + 1 < nb) {
      load_tile(sQ0 + (st ^ 1) * 8192, Q, a.st, (qb + 1) * 64, T, tid, 128);
      load_tile(sO0 + (st ^ 1) * 8192, dO, a.ost, (qb + 1) * 64, T, tid, 128);
      cp_commit();
      if (tid < 64) {
        int i = (qb + 1) * 64 + tid;
        sL[st ^ 1][tid] = (i < T) ? lse[i] * LOG2E : INFINITY;
        sD[st ^ 1][tid] = (i < T) ? Dv[i] : 0.f;
      }
    }
    // S^T[j, i] = K_j . Q_i ;  P^T = exp(S^T * scale - lse_i), masked where i < j
    float p[8][4], dp[8][4];
    zero_acc(p);
    mma_a_tileT(p, kf, sQ, lane);
    zero_acc(dp);
    mma_a_tileT(dp, vf, sO, lane);  // dP^T[j, i] = V_j . dO_i
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int il = nt * 8 + 2 * t4 + (e & 1);
        const int i = qb * 64 + il;
        const int j = j0 + ((e >> 1) << 3);
        float pv = exp2f(p[nt][e] * c2 - sL[st][il]);
        if (i < j) pv = 0.f;
        p[nt][e] = pv;
        dp[nt][e] = pv * (dp[nt][e] - sD[st][il]);  // dS^T
      }
    }
    mma_p_tile(dv, p, sO, lane);   // dV += P^T dO
    mma_p_tile(dk, dp, sQ, lane);  // dK += dS^T Q
    cp_wait_all();
    __syncthreads();
  }
  bf16* dK = static_cast<bf16*>(a.dk) + off;
  bf16* dV = static_cast<bf16*>(a.dv) + off;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int j = j0 + r * 8;
    if (j >= T) continue;
#pragma unroll
    for (int dt = 0; dt < 8; ++dt) {
      *reinterpret_cast<uint32_t*>(dK + (long long)j * a.st + dt * 8 + 2 * t4) =
          pack_bf16(dk[dt][2 * r] * a.scale, dk[dt][2 * r + 1] * a.scale);
      *reinterpret_cast<uint32_t*>(dV + (long long)j * a.st + dt * 8 + 2 * t4) =
          pack_bf16(dv[dt][2 * r], dv[dt][2 * r + 1]);
    }
  }
}

// dQ for a 64-query block: loop over key blocks kb <= qb.
__global__ void __launch_bounds__(128) k_attn_bwd_dq_bf16(AttnArgs a) {
  __shared__ __align__(128) uint8_t smem[8192 * 6];
  const uint32_t sQO = smem_u32(smem);
  const uint32_t sK0 = sQO + 2 * 8192, sV0 = sQO + 4 * 8192;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nqb = gridDim.x;
  const int qb = nqb - 1 - blockIdx.x;
  const int bh = blockIdx.y;
  const int b = bh / a.H, h = bh % a.H;
  const int T = a.T;
  const long long off = b * a.sb + h * a.sh, ooff = b * a.osb + h * a.osh;
  const bf16* Q = static_cast<const bf16*>(a.q) + off;
  const bf16* K = static_cast<const bf16*>(a.k) + off;
  const bf16* Vp = static_cast<const bf16*>(a.v) + off;
  const bf16* dO = static_cast<const bf16*>(a.dO) + ooff;
  const int q0 = qb * 64;
  load_tile(sQO, Q, a.st, q0, T, tid, 128);
  load_tile(sQO + 8192, dO, a.ost, q0, T, tid, 128);
  load_tile(sK0, K, a.st, 0, T, tid, 128);
  load_tile(sV0, Vp, a.st, 0, T, tid, 128);
  cp_commit();
  cp_wait_all();
  __syncthreads();
  uint32_t qf[4][4], of[4][4];
  load_afrag(sQO, warp * 16, lane, qf);
  load_afrag(sQO + 8192, warp * 16, lane, of);
  const int g = lane >> 2, t4 = lane & 3;
  const int i0 = q0 + warp * 16 + g;
  float L2[2], Di[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    int i = i0 + r * 8;
    L2[r] = (i < T) ? a.lse[(long long)bh * T + i] * LOG2E : INFINITY;
    Di[r] = (i < T) ? a.Dbuf[(long long)bh * T + i] : 0.f;
  }
  float dq[8][4];
  zero_acc(dq);
  const float c2 = a.scale * LOG2E;
  for (int kb = 0; kb <= qb; ++kb) {
    const int st = kb & 1;
    const uint32_t sK = sK0 + st * 8192, sV = sV0 + st * 8192;
    if (kb + 1 <= qb) {
      load_tile(sK0 + (st ^ 1) * 8192, K, a.st, (kb + 1) * 64, T, tid, 128);
      load_tile(sV0 + (st ^ 1) * 8192, Vp, a.st, (kb + 1) * 64, T, tid, 128);
      cp_commit();
    }
    float s[8][4], dp[8][4];
    zero_acc(s);
    mma_a_tileT(s, qf, sK, lane);
    zero_acc(dp);
    mma_a_tileT(dp, of, sV, lane);
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = kb * 64 + nt * 8 + 2 * t4 + (e & 1);
        const int r = e >> 1;
        const int i = i0 + r * 8;
        float pv = exp2f(s[nt][e] * c2 - L2[r]);
        if (j > i) pv = 0.f;
        s[nt][e] = pv * (dp[nt][e] - Di[r]);  // dS
      }
    }
    mma_p_tile(dq, s, sK, lane);  // dQ += dS K
    cp_wait_all();
    __syncthreads();
  }
  bf16* dQ = static_cast<bf16*>(a.dq) + off;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int i = i0 + r * 8;
    if (i >= T) continue;
#pragma unroll
    for (int dt = 0; dt < 8; ++dt)
      *reinterpret_cast<uint32_t*>(dQ + (long long)i * a.st + dt * 8 + 2 * t4) =
          pack_bf16(dq[dt][2 * r] * a.scale, dq[dt][2 * r + 1] * a.scale);
  }
}

static bool strides_ok(const AttnArgs& a) {
  return a.d == 64 && a.st % 8 == 0 && a.sh % 8 == 0 && a.sb % 8 == 0 && a.ost % 8 == 0 &&
         a.osh % 8 == 0 && a.osb % 8 == 0;
}

int attn_fwd_bf16(const AttnArgs& a, cudaStream_t s) {
  if (!strides_ok(a)) return (int)cudaErrorInvalidValue;
  dim3 grid((a.T + 63) / 64, a.B * a.H);
  k_attn_fwd_bf16<<<grid, 128, 0, s>>>(a);
  return (int)cudaGetLastError();
}

// D[b, h, i] = sum_c dO[i, c] O[i, c] for d = 64: 8 threads per row, 16 B each.
__global__ void __launch_bounds__(256) k_attn_rowdot64(AttnArgs a) {
  const long long gid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long row = gid >> 3;
  const int part = (int)(gid & 7);
  const long long rows = (long long)a.B * a.H * a.T;
  float s = 0.f;
  if (row < rows) {
    const int i = (int)(row % a.T);
    const int bh = (int)(row / a.T);
    const int b = bh / a.H, h = bh % a.H;
    const long long off = b * a.osb + h * a.osh + (long long)i * a.ost + part * 8;
    float o[8], g[8];
    load16(static_cast<const bf16*>(a.o) + off, o);
    load16(static_cast<const bf16*>(a.dO) + off, g);
#pragma unroll
    for (int e = 0; e < 8; ++e) s += o[e] * g[e];
  }
  s += __shfl_xor_sync(0xffffffffu, s, 1);
  s += __shfl_xor_sync(0xffffffffu, s, 2);
  s += __shfl_xor_sync(0xffffffffu, s, 4);
  if (row < rows && part == 0) a.Dbuf[row] = s;
}

int attn_bwd_bf16(const AttnArgs& a, cudaStream_t s) {
  if (!strides_ok(a)) return (int)cudaErrorInvalidValue;
  long long rows = (long long)a.B * a.H * a.T;
  k_attn_rowdot64<<<(unsigned)((rows * 8 + 255) / 256), 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return (int)e;
  return attn_bwd_tc(a, s);
}

// ------------------------------------------------------------------ fp32 (CUDA cores)
// One warp per query row; each lane takes keys j = lane, lane+32, ...; online
// softmax across 32-key chunks; lanes own output columns c = lane, lane+32, ...
constexpr int kF32MaxD = 128;

__global__ void k_attn_fwd_f32(AttnArgs a) {
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
  k_attn_fwd_f32<<<(unsigned)((rows * 32 + 255) / 256), 256, 0, s>>>(a);
  return (int)cudaGetLastError();
}

int attn_bwd_f32(const AttnArgs& a, cudaStream_t s) {
  if (a.d > kF32MaxD) return (int)cudaErrorInvalidValue;
  long long rows = (long long)a.B * a.H * a.T;
  unsigned grid = (unsigned)((rows * 32 + 255) / 256);
  k_attn_rowdot<float><<<grid, 256, 0, s>>>(a);
  k_attn_bwd_dq_f32<<<grid, 256, 0, s>>>(a);
  k_attn_bwd_dkdv_f32<<<grid, 256, 0, s>>>(a);
  return (int)cudaGetLastError();
}

}  // namespace gpt2k
