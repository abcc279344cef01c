// bf16 GEMM on the 5th-generation tensor cores (tcgen05) for sm_103a.
//
// D[m, n] = sum_k A(m, k) B(n, k), fp32 accumulation in tensor memory.
// Every Linear of the GPT-2 step maps onto it:
//   forward   Y  = X W^T      A = X  (K-major), B = W  (K-major)
//   backward  dX = dY W      A = dY (K-major), B = W  (MN-major)
//             dW = dY^T X    A = dY (MN-major), B = X (MN-major), split over the rows
//
// Structure: persistent clusters of two CTAs (a CTA pair on two SMs), 18 warps
// each; a pair computes 256 x 256 output tiles with the pair MMA (cta_group::2):
//   warp 0      TMA producer of each CTA: its 128 rows of A and its 128 rows of
//               B (half of the tile's 256 N columns), 128-deep k blocks as two
//               128B-swizzled 64-deep slabs, into a 3-stage shared-memory ring;
//               both CTAs' copies complete on the even CTA's barrier of that stage;
//   warp 1      of each CTA allocates 512 TMEM columns (two 128 x 256 fp32
//               accumulators per CTA) together with its peer; one thread of the
//               even CTA issues tcgen05.mma.cta_group::2 (M=256, N=256, K=16) per
//               16-wide k step, reading A and B halves from both CTAs' shared
//               memory and accumulating 128 rows in each CTA's tensor memory, and
//               releases ring stages and finished accumulators in both CTAs with
//               multicast tcgen05.commit;
//   warps 2-17  epilogue of each CTA (its 128 rows of the tile), four warps per
//               TMEM lane quadrant (one per 64-column quarter): tcgen05.ld 32 rows
//               x 16 columns at a time, fused bias /
//               residual / GELU / GELU' / cross-entropy statistics, then the
//               32 x 16 result is staged in 32B-swizzled shared memory and
//               written by a TMA bulk tensor store (coalesced, asynchronous).
//               Residual and GELU' operands arrive the same way, by a TMA load
//               of the matching 32 x 16 box, one chunk ahead.  Sixteen warps
//               (four per SM sub-partition) hide the epilogue's latencies.
// The accumulator double buffer lets the epilogue of tile i overlap the
// mainloop of tile i+1.  Per 64 of K each SM stages 32 KB of operands for a
// 128 x 256 x 64 share of the MMA (a single-CTA 128 x 256 tile stages 48 KB), so
// the operand traffic through L2, TMA and shared memory per flop is a third lower.
// Every wait is bounded (about 2 s of %globaltimer); on expiry the CTA latches
// ST_TIMEOUT in the status word, the other roles stop, outstanding TMA copies and
// MMAs are drained, both CTAs meet at a cluster barrier and TMEM is freed.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace gpt2k {

namespace {
constexpr int BM = 128;       // accumulator rows per CTA
constexpr int PM = 2 * BM;     // rows of a pair tile
constexpr int BN = 256;        // columns of a tile (the pair MMA's N)
constexpr int BNC = BN / 2;    // B rows (output columns) each CTA stages
// A stage holds a 128-deep k block as two 64-deep slabs (the 128B swizzle's width) per
// operand: one wait and one commit of the MMA thread per 8 MMAs.  Its control path runs
// beside 16 busy epilogue warps and costs about 300 cycles per wait / commit round, a
// third of the time at 64-deep stages (512 cycles of MMAs).
constexpr int KS = 64, SLABS = 2, BK = KS * SLABS, STAGES = 3;
constexpr int A_SLAB = BM * KS * 2;   // 16 KB
constexpr int B_SLAB = BNC * KS * 2;  // 16 KB
constexpr int A_TILE = SLABS * A_SLAB;
constexpr int B_TILE = SLABS * B_SLAB;
constexpr int STAGE_BYTES = A_TILE + B_TILE;
constexpr int RING_BYTES = STAGES * STAGE_BYTES;
constexpr int TMEM_COLS = 2 * BN;
constexpr int EPI_WARPS = 16;
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;
constexpr int CW = 16;                          // chunk width: columns per TMEM load
constexpr int WCOLS = BN / (EPI_WARPS / 4);     // columns per epilogue warp and tile (64)
constexpr int NCHUNK = WCOLS / CW;              // chunks per epilogue warp and tile (4)
constexpr int BOX_BYTES = 1024;                 // one staged box: 32 rows x 32 bytes
constexpr int STG_BYTES = 2 * BOX_BYTES;        // per epilogue warp
constexpr int BAR_BYTES = 512;
constexpr int SMEM_BYTES = 1024 + RING_BYTES + EPI_WARPS * STG_BYTES + BAR_BYTES;

struct TcParams {
  GemmArgs g;
  int mt, nt, splits, kps, total_kb;  // mt, nt: pair tiles (256 x 256) along M and N
  uint32_t idesc;
  unsigned* status;
  int poison;
  int out_f32;  // D (or the split-K workspace) holds fp32
  int load_x;   // the epilogue reads a [M, N] bf16 operand (residual or GELU pre-activation)
  int m_fast;   // tile raster: consecutive tiles walk M (sharing a B tile) instead of N
  int a3d, b3d; // MN-major operand loaded by one 3-D box (all its 64-wide blocks) per stage
  int sk;              // schedule with in-kernel partial sums: SK_STREAM or SK_SPLIT (see cta_unit)
  int dp_tiles;        // SK_STREAM: tiles [0, dp_tiles) run whole, one per CTA and wave
  long long sk_iters;  // SK_STREAM: k blocks of tiles [dp_tiles, mt*nt) end to end, cut evenly over the CTAs
  float* sk_part;      // BM x BN fp32 partial-sum slots
  unsigned* sk_flags;  // one ready flag per slot and epilogue warp (zero between launches)
};
enum { SK_NONE = 0, SK_STREAM = 1, SK_SPLIT = 2, SK_REDUCE = 3 };  // SK_REDUCE: host-side plan only

// Tile index -> (M tile, N tile, K split).  Consecutive tiles (one wave of
// CTAs) share the tile of the larger operand, so it is read from DRAM about
// once while the smaller operand is re-read from L2.
__device__ __forceinline__ void tile_coords(const TcParams& p, int tile, int& m_t, int& n_t, int& sp) {
  const int per = p.mt * p.nt;
  sp = tile / per;
  const int r = tile - sp * per;
  if (p.m_fast) {
    m_t = r % p.mt;
    n_t = r / p.mt;
  } else {
    n_t = r % p.nt;
    m_t = r / p.nt;
  }
}

// One CTA's unit of work: k blocks [kb0, kb1) of tile (m_t, n_t), K split sp.
// A U_PART unit leaves its fp32 sums in partial-sum slot `slot`.
enum { U_FULL = 0, U_PART = 1, U_FINISH = 2 };
struct Unit {
  int tile, m_t, n_t, sp, kb0, kb1, role, slot;
};

// Work is dealt to CTA pairs: pair (cluster) c = blockIdx.x / 2 of gridDim.x / 2.
__device__ __forceinline__ int pair_id() { return (int)(blockIdx.x >> 1); }
__device__ __forceinline__ int num_pairs() { return (int)(gridDim.x >> 1); }

// First stream-K iteration of pair c: pair c owns [sk_lo(c), sk_lo(c + 1)).
__device__ __forceinline__ long long sk_lo(const TcParams& p, int c) {
  return p.sk_iters * c / num_pairs();
}

// The u-th unit of this CTA's pair; false past its last.  Both CTAs of a pair
// walk the same units; `slot` is the pair's partial-sum slot (each CTA of the
// pair owns half of it: physical slot 2 * slot + rank).
//   Plain schedule: tiles c, c + P, ... (c = pair, P = pairs) over (split, M tile, N tile).
//   SK_SPLIT: the same walk; split s-1 of a tile (U_FINISH) adds the partial
//   sums that splits 0 .. s-2 (U_PART, slot = their walk index) left for it and
//   runs the epilogue.  The walk is split-major, so one wave of CTAs covers the
//   same K range of many tiles and the operands' k blocks are shared in L2.
//   SK_STREAM: the CTA's share of the stream-K iterations, cut at tile
//   boundaries into fragments, then its whole tiles.  A fragment that reaches
//   the end of its tile (U_FINISH) adds the partial sums that lower CTAs left
//   for that tile and runs the epilogue.  One that does not (U_PART) stores its
//   fp32 sums in the CTA's slot and raises the CTA's flags; only the share's last
//   fragment can be one, and it is taken first, so no CTA's U_PART work ever
//   queues behind a wait on another CTA.
// In both, a U_FINISH unit waits only on U_PART units, which wait on nothing.
__device__ __forceinline__ bool cta_unit(const TcParams& p, int u, Unit& w) {
  int tile;
  const int c = pair_id(), np = num_pairs();
  w.slot = c;
  if (p.sk == SK_STREAM) {
    const int Kb = p.total_kb;
    const long long s = sk_lo(p, c), e = sk_lo(p, c + 1);
    const int nfrag = e > s ? (int)((e - 1) / Kb - s / Kb) + 1 : 0;
    if (u < nfrag) {
      const int i = (e % Kb) != 0 ? (u == 0 ? nfrag - 1 : u - 1) : u;
      const long long t = s / Kb + i;
      const long long lo = t * Kb > s ? t * Kb : s;
      const long long hi = (t + 1) * Kb < e ? (t + 1) * Kb : e;
      w.kb0 = (int)(lo - t * Kb);
      w.kb1 = (int)(hi - t * Kb);
      w.role = w.kb1 < Kb ? U_PART : (w.kb0 > 0 ? U_FINISH : U_FULL);
      tile = p.dp_tiles + (int)t;
    } else {
      tile = c + (u - nfrag) * np;
      if (tile >= p.dp_tiles) return false;
      w.kb0 = 0;
      w.kb1 = Kb;
      w.role = U_FULL;
    }
    tile_coords(p, tile, w.m_t, w.n_t, w.sp);
  } else {
    tile = c + u * np;
    if (tile >= p.mt * p.nt * p.splits) return false;
    tile_coords(p, tile, w.m_t, w.n_t, w.sp);
    w.kb0 = w.sp * p.kps;
    w.kb1 = min(p.total_kb, w.kb0 + p.kps);
    w.role = U_FULL;
    if (p.sk == SK_SPLIT) {
      w.role = w.sp < p.splits - 1 ? U_PART : U_FINISH;
      w.slot = tile;
    }
  }
  w.tile = tile;
  return true;
}

// Stream-K flags and partial sums: gpu-scope release / acquire, L2-only data.
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* f) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(unsigned* f, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}
__device__ __forceinline__ void st_cg4(float* a, const uint32_t* r) {
  asm volatile("st.global.cg.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(a), "r"(r[0]), "r"(r[1]), "r"(r[2]),
               "r"(r[3])
               : "memory");
}
__device__ __forceinline__ float4 ld_cg4(const float* a) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(a)
               : "memory");
  return v;
}
// Warp-collective bounded wait for a flag raised by another CTA (false on
// abort or expiry; expiry latches ST_TIMEOUT).
__device__ __forceinline__ bool flag_wait(const unsigned* f, int lane, volatile int* abort_flag,
                                          unsigned* status) {
  int ok = 1;
  if (lane == 0 && !ld_acquire_gpu(f)) {
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
      if (ld_acquire_gpu(f)) break;
      if (*abort_flag) { ok = 0; break; }
      if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
        if (status) atomicOr(status, ST_TIMEOUT);
        *abort_flag = 1;
        ok = 0;
        break;
      }
      __nanosleep(100);
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) (void)ld_acquire_gpu(f);  // every lane's later reads are ordered after the flag
  return ok != 0;
}


// ------------------------------------------------------------------ epilogue helpers
__device__ __forceinline__ void tma_load_x(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int x,
                                           int y) {
  tma_load_2d(dst, tm, bar, x, y);
}
// One staged box holds 32 rows of 32 bytes in the TMA 32-byte swizzle: the
// 16-byte piece p of row r sits at r*32 + ((p ^ ((r >> 2) & 1)) << 4).  A
// quarter-warp writing the same piece of 8 consecutive rows hits 8 distinct
// 16-byte bank groups.
__device__ __forceinline__ uint32_t box_addr(uint32_t box, int r, int p) {
  return box + (uint32_t)(r * 32 + ((p ^ ((r >> 2) & 1)) << 4));
}
__device__ __forceinline__ void box_store_row(uint32_t box, int r, const uint32_t* w) {
#pragma unroll
  for (int p = 0; p < 2; ++p)
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(box_addr(box, r, p)), "r"(w[4 * p]),
                 "r"(w[4 * p + 1]), "r"(w[4 * p + 2]), "r"(w[4 * p + 3])
                 : "memory");
}
__device__ __forceinline__ void box_load_row_bf16(uint32_t box, int r, float* v) {
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    uint32_t w0, w1, w2, w3;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                 : "r"(box_addr(box, r, p))
                 : "memory");
    const uint32_t w[4] = {w0, w1, w2, w3};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      v[8 * p + 2 * q] = __uint_as_float(w[q] << 16);
      v[8 * p + 2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
    }
  }
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&t);
}
__device__ __forceinline__ void pack16_bf16(const float* v, uint32_t* w) {
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = pack2_bf16(v[2 * j], v[2 * j + 1]);
}

// Column sums of a 32-row x 16-column chunk held one row per lane (v[0..15]):
// four exchange-and-halve shuffle stages leave lane l with column (l >> 1) & 15
// summed over 16 lanes, and a last shuffle adds lane l ^ 1.  Fixed order.
__device__ __forceinline__ float colsum_32x16(const float* v, int lane) {
  float a[8], b[4], c[2];
  const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4, h2 = lane & 2;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float send = h16 ? v[j] : v[j + 8];
    a[j] = (h16 ? v[j + 8] : v[j]) + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float send = h8 ? a[j] : a[j + 4];
    b[j] = (h8 ? a[j + 4] : a[j]) + __shfl_xor_sync(0xffffffffu, send, 8);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float send = h4 ? b[j] : b[j + 2];
    c[j] = (h4 ? b[j + 2] : b[j]) + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  float d = (h2 ? c[1] : c[0]) + __shfl_xor_sync(0xffffffffu, h2 ? c[0] : c[1], 2);
  return d + __shfl_xor_sync(0xffffffffu, d, 1);
}

// 2^x by the hardware approximation (PTX ex2.approx.ftz.f32; relative error about 2^-22).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmD2,
              const __grid_constant__ CUtensorMap tmX, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_tiles = smem_u32(smem);
  const uint32_t s_stg = s_tiles + RING_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + RING_BYTES + EPI_WARPS * STG_BYTES);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], done, xload[EPI_WARPS][2]
  const uint32_t b_full = smem_u32(bars), b_empty = b_full + 8 * STAGES;
  const uint32_t b_tfull = b_empty + 8 * STAGES, b_tempty = b_tfull + 16, b_done = b_tempty + 16;
  const uint32_t b_xload = b_done + 8;
  constexpr int NBARS = 2 * STAGES + 5 + 2 * EPI_WARPS;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + NBARS + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const GemmArgs& g = p.g;
  const uint32_t rank = cluster_ctarank();  // 0: the pair's MMA issuer
  // the even CTA's barriers, as cluster addresses: ring stages fill there, and
  // both CTAs' epilogues hand their accumulator halves back there
  const uint32_t lead_full = mapa_shared(b_full, 0), lead_tempty = mapa_shared(b_tempty, 0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(b_full + 8 * i, 1);  // the even CTA's producer posts both CTAs' bytes
      mbar_init(b_empty + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_tfull + 8 * i, 1);
      mbar_init(b_tempty + 8 * i, 2 * EPI_WARPS);  // one arrival per epilogue warp of either CTA
    }
    mbar_init(b_done, 1);
    for (int i = 0; i < 2 * EPI_WARPS; ++i) mbar_init(b_xload + 8 * i, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmD)) : "memory");
  }
  pdl_wait();  // the predecessor kernel is complete: global memory and TMEM are ours
  if (warp == 1) {  // one warp of each CTA allocates the pair's columns together
    tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(tmem_slot)), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers are initialised and their TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int stage = 0;
      uint32_t phase = 0;
      int last_par[STAGES];
#pragma unroll
      for (int i = 0; i < STAGES; ++i) last_par[i] = -1;
      bool first = true;
      Unit w;
      for (int u = 0; cta_unit(p, u, w); ++u) {
        const int m0 = w.m_t * PM + (int)rank * BM, n0 = w.n_t * BN + (int)rank * BNC;  // this CTA's halves
        bool stop = false;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_wait(b_empty + 8 * stage, phase ^ 1, abort_flag, p.status)) { stop = true; break; }
          if (!((p.poison & POISON_GEMM_TMA) && first)) {
            const uint32_t sa = s_tiles + stage * STAGE_BYTES, sb = sa + A_TILE;
            const uint32_t fb = lead_full + 8 * stage;
            // Only the even CTA arrives, with the byte count of both CTAs' copies (a local
            // arrive: a cluster-scope release per stage from each producer cost about 1,500
            // cycles per k block).  The odd CTA's copies may complete on that barrier before
            // the arrive; the phase cannot complete while the arrive is pending.
            if (rank == 0) mbar_expect_tx(b_full + 8 * stage, 2 * STAGE_BYTES);
            // each 64-deep slab lands in its own region; a slab past K reads zeros
            #pragma unroll
            for (int sl = 0; sl < SLABS; ++sl) {
              const int kk = kb * BK + sl * KS;
              const uint32_t da = sa + sl * A_SLAB, db = sb + sl * B_SLAB;
              if (!g.a_mn) {
                tma_load_2d_pair(da, &tmA, fb, kk, m0);
              } else if (p.a3d) {
                tma_load_3d_pair(da, &tmA, fb, 0, kk, m0 / 64);
              } else {
                tma_load_2d_pair(da, &tmA, fb, m0, kk);
                tma_load_2d_pair(da + 8192, &tmA, fb, m0 + 64, kk);
              }
              if (!g.b_mn) {
                tma_load_2d_pair(db, &tmB, fb, kk, n0);
              } else if (p.b3d) {
                tma_load_3d_pair(db, &tmB, fb, 0, kk, n0 / 64);
              } else {
                tma_load_2d_pair(db, &tmB, fb, n0, kk);
                tma_load_2d_pair(db + 8192, &tmB, fb, n0 + 64, kk);
              }
            }
            last_par[stage] = (int)phase;
          }
          first = false;
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (stop) break;
      }
      // drain: never leave with bulk copies still landing in shared memory.  Both
      // CTAs' copies of a stage complete on the even CTA's barrier, so the even
      // CTA waits for every stage it filled (the odd CTA filled the same ones);
      // the cluster barrier at the end keeps the odd CTA resident until then.
      if (rank == 0) {
#pragma unroll
        for (int i = 0; i < STAGES; ++i)
          if (last_par[i] >= 0) mbar_wait_drain(b_full + 8 * i, (uint32_t)last_par[i]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int abuf = 0;
      uint32_t aphase = 0;
      // Descriptors of stage 0's first k step; another stage, slab or k step only moves the
      // start address (bits 0-13, in 16-byte units, no carry for shared-memory offsets).
      const uint64_t da0 = operand_desc(s_tiles, g.a_mn, 0), db0 = operand_desc(s_tiles + A_TILE, g.b_mn, 0);
      const uint32_t ka = g.a_mn ? 2048 : 32, kb16 = g.b_mn ? 2048 : 32;  // bytes per 16-wide k step
      Unit w;
      for (int u = 0; cta_unit(p, u, w); ++u) {
        const int kb0 = w.kb0, kb1 = w.kb1;
        if (!mbar_wait(b_tempty + 8 * abuf, aphase ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + abuf * BN;
        bool stop = false;
        for (int kb = kb0; kb < kb1; ++kb) {
          // a non-blocking probe first: the stage is usually full already
          if (!mbar_test(b_full + 8 * stage, phase) && !mbar_wait(b_full + 8 * stage, phase, abort_flag, p.status)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint64_t so = (uint64_t)((stage * STAGE_BYTES) >> 4);
          #pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const int sl = k / (KS / 16), ks = k % (KS / 16);
            mma_bf16_pair(d_tmem, da0 + so + ((sl * A_SLAB + ks * ka) >> 4), db0 + so + ((sl * B_SLAB + ks * kb16) >> 4),
                          p.idesc, (kb > kb0 || k > 0) ? 1u : 0u);
          }
          mma_commit_pair_mc(b_empty + 8 * stage, 3);  // the stage is free again in both CTAs
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (stop) break;
        mma_commit_pair_mc(b_tfull + 8 * abuf, 3);  // both halves of the accumulator are ready
        if (++abuf == 2) { abuf = 0; aphase ^= 1; }
      }
      // all MMAs issued by this thread have completed once b_done flips
      mma_commit_pair(b_done);
      mbar_wait_drain(b_done, 0);
    }
  } else {
    // ---------------- epilogue warps 2..17: TMEM lane quadrant warp % 4, column quarter (warp-2)/4
    const int ew = warp - 2, quad = warp & 3, qq = ew >> 2;
    const uint32_t stg = s_stg + ew * STG_BYTES;   // two staged boxes
    const uint32_t xbar = b_xload + 16 * ew;       // their load barriers
    uint32_t xpar = 0;                             // bit b: parity of the next completion of xbar b
    uint32_t xpend = 0;                            // bit b: a load into box b is in flight
    int bx = 0;                                    // box of the current chunk
    bool prev_stored = false;                      // the previous chunk issued a store
    const int epi = g.epi;
    const bool split = p.splits > 1 && p.sk == SK_NONE;  // fp32 partials out, reduced by another kernel
    // chunk c of a tile: rows y = m_t*BM + quad*32 .. +32, columns x = xb + c*CW .. +CW with
    // xb = n_t*BN + qq*WCOLS; this warp's origin of a unit (xb, y), or y = M when the unit
    // stores no output (none left, or a stream-K partial)
    auto warp_origin = [&](bool ok, const Unit& w, int& xb, int& y) {
      if (!ok || w.role == U_PART) { xb = 0; y = g.M; return; }
      xb = w.n_t * BN + qq * WCOLS;
      y = w.m_t * PM + (int)rank * BM + quad * 32;
    };
    // this warp's region of this CTA's half of pair slot j: chunk c, lane l, 16 floats as
    // four float4 at ((c * 4 + q) * 32 + l) * 4
    auto slot_of = [&](int j) {
      return p.sk_part + (size_t)(2 * j + (int)rank) * (BM * BN) + (size_t)ew * (NCHUNK * CW * 32);
    };
    auto flag_of = [&](int j) { return p.sk_flags + (2 * j + (int)rank) * EPI_WARPS + ew; };
    // hand an accumulator buffer back to the MMA issuer (the even CTA)
    auto release_acc = [&](int b) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_remote_arrive(lead_tempty + 8 * b);
    };
    // Prefetch the x operand of the chunk at (x, y) into box b (all lanes track the state).
    auto x_issue = [&](int x, int y, int b) {
      if (!p.load_x || x >= g.N || y >= g.M) return;
      if (lane == 0) {
        bulk_wait_read<0>();  // the last store out of this box has finished reading it
        mbar_expect_tx(xbar + 8 * b, BOX_BYTES);
        tma_load_x(stg + b * BOX_BYTES, &tmX, xbar + 8 * b, x, y);
      }
      xpend |= 1u << b;
    };
    const bool has_bias = epi == EPI_BIAS || epi == EPI_BIAS_RESID || epi == EPI_BIAS_GELU || epi == EPI_BIAS_GELU_H;
    Unit nw;
    bool nok = cta_unit(p, 0, nw);
    int nxb, ny;  // origin of the next unit this warp handles
    warp_origin(nok, nw, nxb, ny);
    x_issue(nxb, ny, 0);
    int abuf = 0;
    uint32_t aphase = 0;
    for (int u = 0; nok; ++u) {
      const Unit w = nw;
      const int m_t = w.m_t, n_t = w.n_t, sp = w.sp;
      const int xb = nxb, y0 = ny;
      nok = cta_unit(p, u + 1, nw);
      warp_origin(nok, nw, nxb, ny);
      // this warp's 64 bias values, two per lane, loaded before the accumulator wait so
      // their latency is hidden; each chunk gathers its 16 with shuffles
      uint32_t bias2 = 0;
      if (has_bias && w.role != U_PART && xb + 2 * lane + 1 < g.N)
        bias2 = __ldg(reinterpret_cast<const unsigned int*>(static_cast<const bf16*>(g.bias) + xb) + lane);
      if (!mbar_wait(b_tfull + 8 * abuf, aphase, abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + ((uint32_t)(quad * 32) << 16) + abuf * BN + qq * WCOLS;
      if (w.role == U_PART) {
        // stream-K partial: fp32 sums to this CTA's slot, then this warp's flag
        float* slot = slot_of(w.slot);
#pragma unroll 1
        for (int c = 0; c < NCHUNK; ++c) {
          uint32_t r[16];
          tmem_ld16(tacc + c * CW, r);
          tmem_ld_wait();
          if (c == NCHUNK - 1) release_acc(abuf);
#pragma unroll
          for (int q = 0; q < 4; ++q) st_cg4(slot + ((c * 4 + q) * 32 + lane) * 4, r + 4 * q);
        }
        __threadfence();
        __syncwarp();
        if (lane == 0 && !(p.poison & POISON_GEMM_FLAG)) st_release_gpu(flag_of(w.slot), 1u);
        x_issue(nxb, ny, bx);  // the next unit's first operand chunk
        prev_stored = false;
        if (++abuf == 2) { abuf = 0; aphase ^= 1; }
        continue;
      }
      // finish: the partial sums of this tile sit in slots ps0 + i * pst, i < pn
      // (SK_STREAM: pairs [j0, this pair), skipping pairs with an empty share;
      // SK_SPLIT: the walk indices of splits 0 .. s-2); wait for each one's flag,
      // then add them in that order
      int ps0 = 0, pn = 0, pst = 1;
      if (w.role == U_FINISH) {
        if (p.sk == SK_STREAM) {
          const long long t0 = (long long)(w.tile - p.dp_tiles) * p.total_kb;
          int j0 = pair_id();
          while (j0 > 0 && sk_lo(p, j0) > t0) --j0;
          ps0 = j0;
          pn = pair_id() - j0;
        } else {
          pst = p.mt * p.nt;
          ps0 = w.tile - (p.splits - 1) * pst;
          pn = p.splits - 1;
        }
        bool ok = true;
        for (int i = 0; i < pn && ok; ++i) {
          const int j = ps0 + i * pst;
          if (p.sk == SK_STREAM && sk_lo(p, j) == sk_lo(p, j + 1)) continue;
          ok = flag_wait(flag_of(j), lane, abort_flag, p.status);
        }
        if (!ok) break;
      }
      const int m = m_t * PM + (int)rank * BM + quad * 32 + lane;
      const int tgt = (epi == EPI_CE && m < g.M) ? g.targets[m] : -1;
      float ce_m = -INFINITY, ce_s = 0.f, ce_t = 0.f;
      bool stop = false;
#pragma unroll 1
      for (int c = 0; c < NCHUNK; ++c) {
        const int b = bx;
        uint32_t r[16];
        tmem_ld16(tacc + c * CW, r);
        tmem_ld_wait();
        if (c == NCHUNK - 1) release_acc(abuf);  // every TMEM read of this accumulator is done
        if (pn) {
          float acc[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[j] = __uint_as_float(r[j]);
          for (int i = 0; i < pn; ++i) {
            const int j = ps0 + i * pst;
            if (p.sk == SK_STREAM && sk_lo(p, j) == sk_lo(p, j + 1)) continue;
            const float* slot = slot_of(j);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 t = ld_cg4(slot + ((c * 4 + q) * 32 + lane) * 4);
              const float2 lo = add2(make_float2(acc[4 * q], acc[4 * q + 1]), make_float2(t.x, t.y));
              const float2 hi = add2(make_float2(acc[4 * q + 2], acc[4 * q + 3]), make_float2(t.z, t.w));
              acc[4 * q] = lo.x; acc[4 * q + 1] = lo.y; acc[4 * q + 2] = hi.x; acc[4 * q + 3] = hi.y;
            }
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(acc[j]);
        }
        // prefetch the next chunk's operand into the other box
        if (c < NCHUNK - 1) x_issue(xb + (c + 1) * CW, y0, b ^ 1);
        else x_issue(nxb, ny, b ^ 1);
        bx ^= 1;
        const int x0 = xb + c * CW;
        if (x0 >= g.N || y0 >= g.M) { prev_stored = false; continue; }
        if (split || epi == EPI_F32) {
          // fp32 result: two 8-column boxes (both staged boxes)
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
          box_store_row(stg, lane, r);
          box_store_row(stg + BOX_BYTES, lane, r + 8);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int z = split ? sp : 0;
            tma_store_3d(&tmD, stg, x0, y0, z);
            if (x0 + 8 < g.N) tma_store_3d(&tmD, stg + BOX_BYTES, x0 + 8, y0, z);
            bulk_commit();
          }
          prev_stored = true;
          continue;
        }
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
        const uint32_t box0 = stg + b * BOX_BYTES;
        if (p.load_x) {
          if (!mbar_wait(xbar + 8 * b, (xpar >> b) & 1u, abort_flag, p.status)) { stop = true; break; }
          xpar ^= 1u << b;
          xpend &= ~(1u << b);
          float xv[16];
          box_load_row_bf16(box0, lane, xv);
          if (epi == EPI_BIAS_RESID) {
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
              const float2 t = add2(make_float2(v[j], v[j + 1]), make_float2(xv[j], xv[j + 1]));
              v[j] = t.x; v[j + 1] = t.y;
            }
          } else {  // EPI_GELU_BWD: dh = da * gelu'(h); EPI_GELU_BWD_H: gelu'(h) from the stored h
            if (epi == EPI_GELU_BWD_H) {
#pragma unroll
              for (int j = 0; j < 16; j += 2) {
                float2 y, dy;
                gelu_and_grad2(make_float2(xv[j], xv[j + 1]), y, dy);
                xv[j] = dy.x; xv[j + 1] = dy.y;
              }
            }
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
              const float2 t = mul2(make_float2(v[j], v[j + 1]), make_float2(xv[j], xv[j + 1]));
              v[j] = t.x; v[j + 1] = t.y;
            }
            if (g.colpart) {  // the bias gradient's partial: this chunk's column sums over 32 rows
              const float cs = colsum_32x16(v, lane);
              const int col = x0 + (lane >> 1);
              if (!(lane & 1) && col < g.N) g.colpart[(size_t)(y0 >> 5) * g.N + col] = cs;
            }
          }
        }
        if (has_bias) {  // columns x0 + 2i, x0 + 2i + 1 sit in lane c * 8 + i (zero past N)
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t bb = __shfl_sync(0xffffffffu, bias2, c * 8 + i);
            const float2 t = add2(make_float2(v[2 * i], v[2 * i + 1]),
                                  make_float2(__uint_as_float(bb << 16), __uint_as_float(bb & 0xFFFF0000u)));
            v[2 * i] = t.x; v[2 * i + 1] = t.y;
          }
        }
        if (epi == EPI_CE) {
          // the logits are rounded to bf16 (pairwise); the stored values feed the statistics
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t t = pack2_bf16(v[2 * j], v[2 * j + 1]);
            v[2 * j] = __uint_as_float(t << 16);
            v[2 * j + 1] = __uint_as_float(t & 0xFFFF0000u);
          }
          const bool full = x0 + CW <= g.V;  // only the last tile of the vocabulary has padding
          float cm = -INFINITY;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (full || x0 + j < g.V) cm = fmaxf(cm, v[j]);
          if (cm > -INFINITY) {
            // e^(z - m) as 2^(z log2(e) - m log2(e)): one fma and one ex2.approx per logit
            constexpr float L2E = 1.4426950408889634f;
            const float mn = fmaxf(ce_m, cm), nml = -mn * L2E;
            float s0 = (ce_m > -INFINITY) ? ce_s * ex2_approx(fmaf(ce_m, L2E, nml)) : 0.f, s1 = 0.f;
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
              if (full || x0 + j < g.V) s0 += ex2_approx(fmaf(v[j], L2E, nml));
              if (full || x0 + j + 1 < g.V) s1 += ex2_approx(fmaf(v[j + 1], L2E, nml));
            }
            ce_m = mn;
            ce_s = s0 + s1;
          }
          if (tgt >= x0 && tgt < x0 + CW) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (x0 + j == tgt) ce_t = v[j];
          }
        }
        uint32_t w[8];
        if (epi == EPI_BIAS_GELU_H) {
          // h rounded to bf16 (D, kept for the backward) and gelu of that rounded h (D2), so a
          // later recompute from D reproduces D2 exactly
          pack16_bf16(v, w);
          float a[16];
          uint32_t wa[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float2 y, dy;
            gelu_and_grad2(make_float2(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xFFFF0000u)), y, dy);
            a[2 * j] = y.x; a[2 * j + 1] = y.y;
          }
          pack16_bf16(a, wa);
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
          box_store_row(stg, lane, w);
          box_store_row(stg + BOX_BYTES, lane, wa);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tmD, stg, x0, y0, 0);
            tma_store_3d(&tmD2, stg + BOX_BYTES, x0, y0, 0);
            bulk_commit();
          }
          prev_stored = true;
          continue;
        }
        if (epi == EPI_BIAS_GELU) {
          // gelu'(h) (D, for the backward) and gelu(h) (D2) from one tanh: both staged boxes
          float a[16];
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            float2 y, dy;
            gelu_and_grad2(make_float2(v[j], v[j + 1]), y, dy);
            a[j] = y.x; a[j + 1] = y.y;
            v[j] = dy.x; v[j + 1] = dy.y;
          }
          pack16_bf16(v, w);
          uint32_t wa[8];
          pack16_bf16(a, wa);
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
          box_store_row(stg, lane, w);
          box_store_row(stg + BOX_BYTES, lane, wa);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tmD, stg, x0, y0, 0);
            tma_store_3d(&tmD2, stg + BOX_BYTES, x0, y0, 0);
            bulk_commit();
          }
          prev_stored = true;
          continue;
        }
        pack16_bf16(v, w);
        if (!p.load_x) {
          // box b was last read by the store two chunks back (or one, if the last chunk stored nothing)
          if (lane == 0) {
            if (prev_stored) bulk_wait_read<1>();
            else bulk_wait_read<0>();
          }
          __syncwarp();
        }
        box_store_row(box0, lane, w);  // with load_x: in place over this row's operand
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tmD, box0, x0, y0, 0);
          bulk_commit();
        }
        prev_stored = true;
      }
      if (stop) break;
      if (pn) {  // the partial sums are consumed: lower the flags for the next launch
        __syncwarp();
        if (lane == 0)
          for (int i = 0; i < pn; ++i) *flag_of(ps0 + i * pst) = 0u;
      }
      // one statistics partial per row and WCOLS-column quarter tile that starts inside N
      if (epi == EPI_CE && !split && m < g.M && n_t * BN + qq * WCOLS < g.N) {
        const int part = n_t * (BN / WCOLS) + qq;
        g.ce_max[(long long)m * g.ce_ld + part] = ce_m;
        g.ce_sum[(long long)m * g.ce_ld + part] = ce_s;
        const int c0 = n_t * BN + qq * WCOLS;
        if (tgt >= c0 && tgt < c0 + WCOLS) g.ce_tgt[m] = ce_t;
      }
      if (++abuf == 2) { abuf = 0; aphase ^= 1; }
    }
    // never leave with bulk copies still reading or filling this warp's boxes (the stores'
    // global writes complete with the kernel; only the reads of shared memory must be done)
    if (lane == 0) bulk_wait_read<0>();
    for (int b = 0; b < 2; ++b)
      if (xpend & (1u << b)) mbar_wait_drain(xbar + 8 * b, (xpar >> b) & 1u);
    __syncwarp();
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  // neither CTA leaves while its peer may still signal its barriers or read its
  // shared memory; then each frees the pair's columns
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*PFN_encodeTiled_t)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                      const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                      const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                      CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

PFN_encodeTiled_t get_encode() {
  static PFN_encodeTiled_t fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled_t>(ptr);
  }
  return fn;
}

// 2-D bf16 operand map over a row-major [outer, inner] matrix with leading
// dimension ld (elements), 128-byte swizzle (the MMA's operand layout).
bool make_tmap(CUtensorMap* tm, const void* base, long long inner, long long outer, long long ld,
               int box_inner, int box_outer) {
  PFN_encodeTiled_t enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// MN-major operand map over a row-major [K, MN] matrix (leading dimension ld,
// MN % 64 == 0) seen as 3-D (64 MN elements, K rows, MN / 64 blocks): one box of
// 64 x 64 x nblk lands as nblk consecutive 8 KB blocks of 64 K rows x 128 bytes,
// the layout the MMA descriptors expect (128B swizzle).
bool make_tmap_mn3d(CUtensorMap* tm, const void* base, long long mn, long long k, long long ld, int nblk) {
  PFN_encodeTiled_t enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {64, (cuuint64_t)k, (cuuint64_t)(mn / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, 128};
  cuuint32_t box[3] = {64, 64, (cuuint32_t)nblk};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                   es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Epilogue box map: [depth][rows][cols] with leading dimension ld (elements) and
// depth stride rows*ld, boxes of 32 bytes x 32 rows x 1, 32-byte swizzle.
bool make_box_map(CUtensorMap* tm, const void* base, int f32, long long cols, long long rows,
                  long long depth, long long ld) {
  PFN_encodeTiled_t enc = get_encode();
  if (!enc) return false;
  const int es = f32 ? 4 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)depth};
  cuuint64_t strides[2] = {(cuuint64_t)ld * es, (cuuint64_t)ld * es * rows};
  cuuint32_t box[3] = {(cuuint32_t)(32 / es), 32, 1};
  cuuint32_t el[3] = {1, 1, 1};
  CUresult r = enc(tm, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, el, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D bf16 epilogue operand map (residual / gelu'): 32 rows x 16 columns, 32-byte swizzle.
bool make_x_map(CUtensorMap* tm, const void* base, long long cols, long long rows, long long ld) {
  PFN_encodeTiled_t enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {16, 32};
  cuuint32_t el[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                   el, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

int gemm_tc_stat_cols() { return WCOLS; }

// CTA pairs of k_gemm_tc that can be resident at once on the current device
// (queried once per device and context; at most half the SMs).
static PerDeviceOnce g_smem_attr;  // k_gemm_tc's shared-memory limit, set per device and context

static int gemm_pairs() {
  static PerDeviceOnce once;
  static int pairs[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms() / 2;
  const unsigned long long id = current_context_id();
  if (id != 0 && once.ctx[dev] == id && pairs[dev] > 0) return pairs[dev];
  int n = 0;
  if (smem_limit_once(reinterpret_cast<const void*>(k_gemm_tc), SMEM_BYTES, &g_smem_attr) != cudaSuccess)
    (void)cudaGetLastError();
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = launch_cfg(dim3(2), dim3(NUM_THREADS), SMEM_BYTES, nullptr, attr, true);
  if (cudaOccupancyMaxActiveClusters(&n, k_gemm_tc, &cfg) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    n = num_sms() / 2;
  }
  if (n > num_sms() / 2) n = num_sms() / 2;
  pairs[dev] = n;
  once.ctx[dev] = current_context_id();
  return n;
}

int gemm_tc_pairs() { return gemm_pairs(); }

size_t gemm_tc_ws_bytes(int M, int N, int splits) {
  return splits > 1 ? (size_t)splits * M * N * sizeof(float) : 0;
}

// Partial-sum slots of the in-kernel schedules: three per SM (a pair slot is two
// of them, one per CTA).
static int sk_slots() { return 3 * num_sms(); }
static size_t sk_flag_bytes() { return ((size_t)sk_slots() * EPI_WARPS * 4 + 1023) / 1024 * 1024; }

size_t gemm_tc_sk_ws_bytes() { return sk_flag_bytes() + (size_t)sk_slots() * BM * BN * sizeof(float); }
size_t gemm_tc_sk_plane_offset() { return sk_flag_bytes(); }

int gemm_tc_pick_splits(int M, int N, int K, int sms) {  // sms: CTA pairs
  const int tiles = ((M + PM - 1) / PM) * ((N + BN - 1) / BN);
  const int total_kb = (K + BK - 1) / BK;
  if (tiles >= sms) return 1;
  int best = 1;
  double best_score = -1.0;
  for (int s = 1; s <= 16; ++s) {
    const int kps = (total_kb + s - 1) / s;
    if (s > 1 && kps * BK < 256) break;  // at least 256 of K per split
    const int work = tiles * s;
    const int waves = (work + sms - 1) / sms;
    const double eff = (double)work / ((double)waves * sms);
    const double score = eff - 0.02 * s;
    if (score > best_score) { best_score = score; best = s; }
  }
  return best;
}

int gemm_tc_effective_splits(int K, int splits) {
  const int total_kb = (K + BK - 1) / BK;
  if (splits < 1) splits = 1;
  if (splits > total_kb) splits = total_kb;
  const int kps = (total_kb + splits - 1) / splits;
  return (total_kb + kps - 1) / kps;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Schedule for T pair tiles of Kb k blocks on G CTA pairs (GEMM_TC_STREAM_K):
//  - T >= G, last wave part-empty by more than 3%, tiles at least 2048 deep in
//    K: SK_STREAM over the leftover tiles (whole waves stay data-parallel).
//    Shallower tiles are epilogue-bound; cutting them adds epilogues, not speed.
//  - T < G: s = the split count of gemm_tc_pick_splits.  Two splits: SK_SPLIT
//    (the second split adds the first's sums).  More: the finishing CTAs would
//    each read s - 1 partial tiles while the rest idle, so the splits write fp32
//    planes into the slot area and a separate kernel reduces them over all SMs
//    (SK_REDUCE; plain-store epilogues whose planes fit), else SK_SPLIT.
// `force` (GEMM_TC_STREAM_K_FORCE) takes SK_STREAM whenever T % G != 0.
static int sk_plan(const GemmArgs& g, int T, int Kb, int G, bool force, int& dp, int& skt, int& splits) {
  const int M = g.M, N = g.N, K = g.K;
  const int rem = T % G;
  if (force) {
    if (T >= G && rem == 0) return SK_NONE;
    dp = T >= G ? T - rem : 0;
    skt = T >= G ? rem : T;
    return SK_STREAM;
  }
  if (T >= G) {
    if (rem == 0 || Kb * BK < 2048) return SK_NONE;
    const double eff = (double)T / ((double)(T / G + 1) * G);
    if (eff >= 0.97) return SK_NONE;
    dp = T - rem;
    skt = rem;
    return SK_STREAM;
  }
  const int s = gemm_tc_effective_splits(K, gemm_tc_pick_splits(M, N, K, G));
  if (s < 2) return SK_NONE;
  splits = s;
  if (s > 2 && (g.epi == EPI_STORE || g.epi == EPI_F32) &&
      gemm_tc_ws_bytes(M, N, s) <= (size_t)sk_slots() * BM * BN * sizeof(float))
    return SK_REDUCE;
  if (2LL * (s - 1) * T > sk_slots()) return SK_NONE;
  return SK_SPLIT;
}

int gemm_tc(const GemmArgs& g, int splits, void* ws, size_t ws_bytes, unsigned* status,
            cudaStream_t s, int reduce, int* reduce_splits) {
  if (reduce_splits) *reduce_splits = 0;
  if (g.M <= 0 || g.N <= 0 || g.K <= 0) return (int)cudaErrorInvalidValue;
  if (g.N % 8 || g.lda % 8 || g.ldb % 8 || g.ldd % 8) return (int)cudaErrorInvalidValue;
  if (!aligned16(g.A) || !aligned16(g.B) || !aligned16(g.D)) return (int)cudaErrorInvalidValue;
  if (g.epi == EPI_BIAS_RESID && (g.ldr % 8 || !aligned16(g.resid))) return (int)cudaErrorInvalidValue;
  const bool gelu_fwd = g.epi == EPI_BIAS_GELU || g.epi == EPI_BIAS_GELU_H;
  const bool gelu_bwd = g.epi == EPI_GELU_BWD || g.epi == EPI_GELU_BWD_H;
  if (gelu_bwd && (g.ldaux % 8 || !aligned16(g.aux))) return (int)cudaErrorInvalidValue;
  if (gelu_fwd && !aligned16(g.D2)) return (int)cudaErrorInvalidValue;
  if ((g.epi == EPI_BIAS || g.epi == EPI_BIAS_RESID || gelu_fwd) && !aligned16(g.bias))
    return (int)cudaErrorInvalidValue;
  cudaError_t ae = smem_limit_once(reinterpret_cast<const void*>(k_gemm_tc), SMEM_BYTES, &g_smem_attr);
  if (ae != cudaSuccess) return (int)ae;
  TcParams p;
  p.g = g;
  p.mt = (g.M + PM - 1) / PM;
  p.nt = (g.N + BN - 1) / BN;
  p.total_kb = (g.K + BK - 1) / BK;
  p.sk = 0;
  p.dp_tiles = 0;
  p.sk_iters = 0;
  p.sk_part = nullptr;
  p.sk_flags = nullptr;
  if (splits == GEMM_TC_STREAM_K || splits == GEMM_TC_STREAM_K_FORCE) {
    if (!ws || !aligned16(ws) || ws_bytes < gemm_tc_sk_ws_bytes()) return (int)cudaErrorInvalidValue;
    int dp = 0, skt = 0, ssplit = 1;
    const int plan = sk_plan(g, p.mt * p.nt, p.total_kb, gemm_pairs(), splits == GEMM_TC_STREAM_K_FORCE, dp, skt,
                             ssplit);
    char* slots = static_cast<char*>(ws) + sk_flag_bytes();
    if (plan == SK_REDUCE) {  // plain split-K into the slot area
      ws = slots;
      ws_bytes = (size_t)sk_slots() * BM * BN * sizeof(float);
      splits = ssplit;
      if (reduce_splits && !reduce) *reduce_splits = ssplit;
    } else {
      p.sk = plan;
      if (p.sk != SK_NONE) {
        p.dp_tiles = dp;
        p.sk_iters = (long long)skt * p.total_kb;
        p.sk_flags = static_cast<unsigned*>(ws);
        p.sk_part = reinterpret_cast<float*>(slots);
      }
      splits = p.sk == SK_SPLIT ? ssplit : 1;
    }
  }
  if (splits < 1) splits = 1;
  if (splits > p.total_kb) splits = p.total_kb;
  p.kps = (p.total_kb + splits - 1) / splits;
  p.splits = (p.total_kb + p.kps - 1) / p.kps;
  if (p.splits > 1 && p.sk == SK_NONE) {
    if (g.epi != EPI_STORE && g.epi != EPI_F32) return (int)cudaErrorInvalidValue;
    if (!ws || !aligned16(ws) || ws_bytes < gemm_tc_ws_bytes(g.M, g.N, p.splits))
      return (int)cudaErrorInvalidValue;
  }
  p.status = status;
  p.poison = test_poison();
  p.out_f32 = ((p.splits > 1 && p.sk == SK_NONE) || g.epi == EPI_F32) ? 1 : 0;
  p.load_x = (g.epi == EPI_BIAS_RESID || gelu_bwd) ? 1 : 0;
  p.m_fast = ((double)g.N * g.K > (double)g.M * g.K) ? 1 : 0;
  CUtensorMap tmA, tmB, tmD, tmD2, tmX;
  p.a3d = (g.a_mn && g.M % 64 == 0) ? 1 : 0;
  p.b3d = (g.b_mn && g.N % 64 == 0) ? 1 : 0;
  bool ok = p.a3d ? make_tmap_mn3d(&tmA, g.A, g.M, g.K, g.lda, BM / 64)
                  : g.a_mn ? make_tmap(&tmA, g.A, g.M, g.K, g.lda, 64, 64)
                           : make_tmap(&tmA, g.A, g.K, g.M, g.lda, 64, BM);
  ok = ok && (p.b3d ? make_tmap_mn3d(&tmB, g.B, g.N, g.K, g.ldb, BNC / 64)
                    : g.b_mn ? make_tmap(&tmB, g.B, g.N, g.K, g.ldb, 64, 64)
                             : make_tmap(&tmB, g.B, g.K, g.N, g.ldb, 64, BNC));
  if (p.splits > 1 && p.sk == SK_NONE)
    ok = ok && make_box_map(&tmD, ws, 1, g.N, g.M, p.splits, g.N);
  else
    ok = ok && make_box_map(&tmD, g.D, p.out_f32, g.N, g.M, 1, g.ldd);
  if (gelu_fwd)
    ok = ok && make_box_map(&tmD2, g.D2, 0, g.N, g.M, 1, g.ldd);
  else
    tmD2 = tmD;
  if (g.epi == EPI_BIAS_RESID)
    ok = ok && make_x_map(&tmX, g.resid, g.N, g.M, g.ldr);
  else if (gelu_bwd)
    ok = ok && make_x_map(&tmX, g.aux, g.N, g.M, g.ldaux);
  else
    tmX = tmA;
  if (!ok) return (int)cudaErrorInvalidValue;
  // kind::f16 instruction descriptor: D fp32, A/B bf16, operand majors, N >> 3, M >> 4
  // (the pair MMA: M = 256 rows, 128 from each CTA)
  p.idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)g.a_mn << 15) |
            ((uint32_t)g.b_mn << 16) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(PM >> 4) << 24);
  const int ntiles = p.mt * p.nt * p.splits;
  int pairs = gemm_pairs();  // a stream-K launch spreads its iterations over every pair
  if (p.sk != SK_STREAM && pairs > ntiles) pairs = ntiles;
  launch_k_pair(k_gemm_tc, 2 * pairs, NUM_THREADS, SMEM_BYTES, s, tmA, tmB, tmD, tmD2, tmX, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return (int)e;
  if (p.splits > 1 && p.sk == SK_NONE && reduce) {
    splitk_reduce(g.D, g.epi == EPI_F32, g.ldd, static_cast<float*>(ws), p.splits, g.M, g.N, s);
    e = cudaGetLastError();
  }
  return (int)e;
}

}  // namespace gpt2k
