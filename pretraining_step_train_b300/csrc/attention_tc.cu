// Causal attention on the 5th-generation tensor cores (tcgen05) for sm_103a,
// d = 64, never materialising the T x T score matrix (online softmax over
// 128-key tiles, FlashAttention-style: "Let's reproduce GPT-2 (124M)" wiki
// page, "GPU optimisation ladder").
//
// Forward: persistent, one CTA per SM walks work items (a pair of adjacent
// 128-query tiles of one (batch, head)), heaviest first, item c, c + grid, ...
//   warp 0      TMA: the item's two Q tiles, then K and V tiles of 128 keys into
//               a 4-stage ring that runs on across items (4-D tensor maps over
//               the strided q / k / v views, 128B swizzle; rows past T are zeros);
//   warp 1      owns 512 TMEM columns: per query tile t an S buffer (128 fp32
//               columns), the O accumulator (64) and a P buffer (64 columns of
//               bf16 pairs);
//   warps 1, 2  MMA issuers: warp 1 issues S_t = Q_t K_j^T (M=128, N=128, K=64) for
//               both query tiles, warp 2 O_t += P_t V_j (M=128, N=64, K=128, A from
//               TMEM); each product goes as soon as its own inputs are ready, and an S
//               never waits behind PV issue, so the tensor core works on one tile's
//               products while the softmax warps work on the other's;
//   warps 4-7   softmax of query tile 0, warps 8-11 of tile 1 (warp 3 idles): each
//               thread owns one query row (lane quadrant = warp % 4) and all 128
//               keys of a tile, so the row max and sum stay in the thread; p =
//               2^(s*scale*log2e - m) (ex2.approx: 32 per cycle per SM, so the
//               32K exponentials of a key tile take fewer cycles than its MMAs);
//               O is rescaled in TMEM only when the running max has to move by
//               more than 2^8; P (bf16 pairs) goes to TMEM for the PV MMA.
// Epilogue: O / l -> bf16 rows, lse = (m + log2 l) ln 2 (natural log).
// Every wait is bounded; on expiry the CTA latches ST_TIMEOUT (when a status
// word is given), drains its copies and MMAs, frees TMEM and returns.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace gpt2k {

namespace {

constexpr int AT_B = 128;                       // queries per tile = keys per tile
constexpr int AT_D = 64;                        // head size
constexpr int AT_TILE = AT_B * AT_D * 2;        // 16 KB: one [128 x 64] bf16 tile
constexpr int AT_THREADS = 384;
constexpr int AT_TMEM_COLS = 512;
// forward: smem two sets of (Q_0 | Q_1) (a Q_t tile then stages tile t's O for its tensor
// store) | K,V ring; TMEM S_t at 128 t, O_t at 256 + 64 t, P_t at 384 + 64 t
constexpr int FW_STAGES = 4;
constexpr int FW_Q = 0, FW_KV = 4 * AT_TILE;  // Q set q: tile t at FW_Q + (2 q + t) TILE; stage s: K at FW_KV + 2 s TILE, V after
constexpr int FW_BAR = FW_KV + 2 * FW_STAGES * AT_TILE;
constexpr int FW_NBARS = 4 + 2 * FW_STAGES + 8 + 1 + 2;
constexpr int AT_SMEM = 1024 + FW_BAR + 8 * (FW_NBARS + 2);
constexpr uint32_t FW_S_COL = 0, FW_O_COL = 256, FW_P_COL = 384;
constexpr int FW_REGS_LAUNCH = 168, FW_REGS_CTRL = 64, FW_REGS_SOFTMAX = 216;
static_assert(128 * FW_REGS_CTRL + 256 * FW_REGS_SOFTMAX <= AT_THREADS * FW_REGS_LAUNCH,
              "the register split must fit in the launch's registers");

struct AtParams {
  AttnArgs a;
  int nq;        // query tiles per (batch, head)
  int nqp;       // query-tile pairs per (batch, head): ceil(nq / 2)
  int swap_ht;   // the q / k / v tensor maps index (d, h, t, b) instead of (d, t, h, b)
  int swap_o;    // the same for the o tensor map
  float c2;      // scale * log2(e)
  uint32_t idesc_s, idesc_pv;
  unsigned* status;
  int poison;  // test hook (POISON_ATTN_FWD): the producer skips its first K/V stage
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&t);
}
// Bounded mbarrier wait taken by every lane, with a warp-uniform outcome.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned* status) {
  const bool ok = mbar_wait(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}
// One arrival for the warp once every lane's prior work is done.
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}
// Three-input fp32 max (one instruction on sm_100+).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Max of 128 values in four independent chains (short dependency depth).
__device__ __forceinline__ float row_max128(const float* v) {
  float m[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
  for (int i = 4; i < 128; i += 8) {
    m[0] = max3(m[0], v[i], v[i + 1]);
    m[1] = max3(m[1], v[i + 2], v[i + 3]);
    m[2] = max3(m[2], v[i + 4], v[i + 5]);
    m[3] = max3(m[3], v[i + 6], v[i + 7]);
  }
  return max3(m[0], m[1], fmaxf(m[2], m[3]));
}

// Stores 16-byte piece c (0..7) of row r of a [128 x 128 B] tile with the 128B swizzle
// (piece c of row r sits at r * 128 + ((c ^ (r & 7)) << 4)), as TMA reads and writes it.
__device__ __forceinline__ void st_swizzled(uint32_t tile, int r, int c, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(tile + (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4))),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__global__ void __launch_bounds__(AT_THREADS, 1)
    k_attn_fwd_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
              const AtParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + FW_BAR);
  // q_full[2], q_empty[2] (per Q set), kv_full[4], kv_empty[4], s_full[2], s_empty[2], p_full[2],
  // pv_done[2] (per query tile), done
  const uint32_t b_qf = smem_u32(bars), b_qe = b_qf + 16, b_kvf = b_qe + 16, b_kve = b_kvf + 8 * FW_STAGES;
  const uint32_t b_sf = b_kve + 8 * FW_STAGES, b_se = b_sf + 16, b_pf = b_se + 16, b_pv = b_pf + 16;
  const uint32_t b_done = b_pv + 16, b_stg = b_done + 8;  // staged[2]: a tile's O rows are in shared memory
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + FW_NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + FW_NBARS + 1);

  const AttnArgs& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BH = a.B * a.H;
  const int nitems = p.nqp * BH;
  // work item w: query tiles 2 qp and 2 qp + 1 with qp = nqp-1 - w / BH (heaviest first),
  // (batch, head) = w % BH; the second tile is absent when 2 qp + 1 = nq.  Tile 0 uses
  // key tiles 0 .. 2 qp, tile 1 key tiles 0 .. 2 qp + 1.

  if (threadIdx.x == 0) {
    for (int q = 0; q < 2; ++q) {
      mbar_init(b_qf + 8 * q, 1);
      // the S issuer's commit after the item's last S, and per query tile the thread whose
      // tensor store of the tile's O has read its Q tile (tile 0's twice when the item has no
      // tile 1)
      mbar_init(b_qe + 8 * q, 3);
    }
    for (int i = 0; i < FW_STAGES; ++i) {
      mbar_init(b_kvf + 8 * i, 1);
      mbar_init(b_kve + 8 * i, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(b_sf + 8 * t, 1);
      mbar_init(b_se + 8 * t, 4);  // one arrival per softmax warp of the tile
      mbar_init(b_pf + 8 * t, 4);
      mbar_init(b_pv + 8 * t, 1);
    }
    mbar_init(b_done, 2);  // one commit per issuer
    for (int t = 0; t < 2; ++t) mbar_init(b_stg + 8 * t, 4);  // one arrival per softmax warp of the tile
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  pdl_wait();  // the predecessor kernel is complete: global memory and TMEM are ours
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), AT_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // registers: 384 threads x 168 at launch = 64512; warps 0-3 keep 64, the softmax
  // warpgroups take 216 (128 x 64 + 256 x 216 = 63488)
  if (warp < 4) {
    regs_lower<FW_REGS_CTRL>();
    if (warp == 0) {
      if (lane == 0) {
        // ---------------- TMA producer
        int last_par[FW_STAGES] = {-1, -1, -1, -1}, q_par[2] = {-1, -1};
        int g = 0;  // K/V tiles issued so far (ring position)
        bool ok = true;
        for (int w = blockIdx.x, it = 0; ok && w < nitems; w += gridDim.x, ++it) {
          const int qp = p.nqp - 1 - w / BH, bh = w % BH, b = bh / a.H, h = bh % a.H;
          const bool has1 = 2 * qp + 1 < p.nq;
          const int nk = 2 * qp + (has1 ? 2 : 1);
          auto load = [&](const CUtensorMap* tm, uint32_t dst, uint32_t bar, int t0) {
            if (p.swap_ht) tma_load_4d(dst, tm, bar, 0, h, t0, b);
            else tma_load_4d(dst, tm, bar, 0, t0, h, b);
          };
          // Q set it % 2 was last read by the S MMAs of item it - 2
          const int qs = it & 1;
          if (it >= 2 && !mbar_wait(b_qe + 8 * qs, (uint32_t)((it - 2) >> 1) & 1u, abort_flag, p.status)) break;
          mbar_expect_tx(b_qf + 8 * qs, (has1 ? 2 : 1) * AT_TILE);
          load(&tmQ, sbase + FW_Q + 2 * qs * AT_TILE, b_qf + 8 * qs, 2 * qp * AT_B);
          if (has1) load(&tmQ, sbase + FW_Q + (2 * qs + 1) * AT_TILE, b_qf + 8 * qs, (2 * qp + 1) * AT_B);
          q_par[qs] = (it >> 1) & 1;
          for (int j = 0; j < nk; ++j, ++g) {
            const int st = g % FW_STAGES;
            const uint32_t ph = (uint32_t)(g / FW_STAGES) & 1u;
            if (!mbar_wait(b_kve + 8 * st, ph ^ 1u, abort_flag, p.status)) { ok = false; break; }
            if ((p.poison & POISON_ATTN_FWD) && g == 0) continue;
            const uint32_t kd = sbase + FW_KV + st * 2 * AT_TILE;
            mbar_expect_tx(b_kvf + 8 * st, 2 * AT_TILE);
            load(&tmK, kd, b_kvf + 8 * st, j * AT_B);
            load(&tmV, kd + AT_TILE, b_kvf + 8 * st, j * AT_B);
            last_par[st] = (int)ph;
          }
        }
        // never leave with copies still landing in shared memory
        for (int q = 0; q < 2; ++q)
          if (q_par[q] >= 0) mbar_wait_drain(b_qf + 8 * q, (uint32_t)q_par[q]);
        for (int i = 0; i < FW_STAGES; ++i)
          if (last_par[i] >= 0) mbar_wait_drain(b_kvf + 8 * i, (uint32_t)last_par[i]);
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // ---------------- S issuer: S_t(j) = Q_t K_j^T for both query tiles, in the order
        // S_0(0), S_1(0), S_0(1), S_1(1), ...; S_t(j) once K_j has landed and tile t's
        // warps have read S_t(j-1).  The PV products come from another thread: an MMA issue
        // blocks while the tensor core is busy, and S_t(j+1) must not sit behind the PV
        // issue of the previous key tile (its tile would wait for it).
        int cnt_s[2] = {0, 0};  // S products issued per tile, all items
        bool ok = true;
        int g = 0;  // ring position of the item's key tile 0
        for (int w = blockIdx.x, it = 0; ok && w < nitems; w += gridDim.x, ++it) {
          const int qt0 = 2 * (p.nqp - 1 - w / BH);
          const bool has1 = qt0 + 1 < p.nq;
          const int nk_item = qt0 + (has1 ? 2 : 1);  // tile t uses key tiles 0 .. qt0 + t
          const int qs = it & 1;
          if (!mbar_wait(b_qf + 8 * qs, (uint32_t)(it >> 1) & 1u, abort_flag, p.status)) break;
          for (int j = 0; ok && j < nk_item; ++j) {
            const int st = (g + j) % FW_STAGES;
            if (!mbar_wait(b_kvf + 8 * st, (uint32_t)((g + j) / FW_STAGES) & 1u, abort_flag, p.status)) {
              ok = false;
              break;
            }
            const uint32_t kd = sbase + FW_KV + st * 2 * AT_TILE;
            for (int t = 0; t < 2; ++t) {
              if (j > qt0 + t || (t == 1 && !has1)) continue;
              if (cnt_s[t] > 0 && !mbar_wait(b_se + 8 * t, (uint32_t)(cnt_s[t] - 1) & 1u, abort_flag, p.status)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t qd = sbase + FW_Q + (2 * qs + t) * AT_TILE;
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_bf16(tmem + FW_S_COL + 128 * t, operand_desc(qd, 0, k), operand_desc(kd, 0, k), p.idesc_s,
                         k > 0 ? 1u : 0u);
              mma_commit(b_sf + 8 * t);
              ++cnt_s[t];
            }
          }
          if (ok) mma_commit(b_qe + 8 * qs);  // no product reads the item's Q set any more
          g += nk_item;
        }
        // every product issued by either issuer has completed once b_done flips
        mma_commit(b_done);
        mbar_wait_drain(b_done, 0);
      }
    } else if (warp == 2) {
      if (lane == 0) {
        // ---------------- PV issuer: O_t += P_t(j) V_j once tile t's warps have written
        // P_t(j), in the order PV_0(0), PV_1(0), PV_0(1), ...  After key tile j's last PV its
        // commit releases K_j / V_j's ring stage (the S products that read K_j were complete
        // before any P_t(j) could be formed).
        int cnt_pv[2] = {0, 0};  // PV products issued per tile, all items
        bool ok = true;
        int g = 0;
        for (int w = blockIdx.x; ok && w < nitems; w += gridDim.x) {
          const int qt0 = 2 * (p.nqp - 1 - w / BH);
          const bool has1 = qt0 + 1 < p.nq;
          const int nk_item = qt0 + (has1 ? 2 : 1);
          for (int j = 0; ok && j < nk_item; ++j) {
            const int st = (g + j) % FW_STAGES;
            const uint32_t vd = sbase + FW_KV + st * 2 * AT_TILE + AT_TILE;
            for (int t = 0; t < 2; ++t) {
              if (j > qt0 + t || (t == 1 && !has1)) continue;
              if (!mbar_wait(b_pf + 8 * t, (uint32_t)cnt_pv[t] & 1u, abort_flag, p.status)) {
                ok = false;
                break;
              }
              tc_fence_after();
              // A = P_t in TMEM: 16 keys per MMA = 8 columns of bf16 pairs
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_bf16_tmem_a(tmem + FW_O_COL + 64 * t, tmem + FW_P_COL + 64 * t + kk * 8,
                                operand_desc(vd, 1, kk), p.idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
              mma_commit(b_pv + 8 * t);
              ++cnt_pv[t];
            }
            if (ok) mma_commit(b_kve + 8 * st);
          }
          g += nk_item;
        }
        mma_commit(b_done);
        mbar_wait_drain(b_done, 0);
      }
    }
  } else {
    regs_raise<FW_REGS_SOFTMAX>();
    // ---------------- softmax warps: query tile t = (warp - 4) / 4, lane quadrant warp % 4
    const int t = (warp - 4) >> 2, quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t s_col = FW_S_COL + 128 * t, o_col = FW_O_COL + 64 * t, p_col = FW_P_COL + 64 * t;
    const uint32_t b_sft = b_sf + 8 * t, b_set = b_se + 8 * t, b_pft = b_pf + 8 * t, b_pvt = b_pv + 8 * t;
    const float2 c2 = make_float2(p.c2, p.c2);
    bool ok = true;
    int n_s = 0, n_pv = 0;  // S tiles read and PV MMAs waited for, by this tile's warps
    int n_it = 0;           // items of this tile so far
    int pend = -1, pend_n = 0;  // quad-0 warp: the Q set whose O store is in flight, arrivals owed
    for (int w = blockIdx.x, it = 0; ok && w < nitems; w += gridDim.x, ++it) {
      const int qp = p.nqp - 1 - w / BH, bh = w % BH, b = bh / a.H, h = bh % a.H;
      const int qt = 2 * qp + t;
      if (qt >= p.nq) continue;  // this item has no second tile
      const bool has1 = 2 * qp + 1 < p.nq;
      const int qs = it & 1;
      const int nk = qt + 1;
      const int qi = qt * AT_B + r;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nk; ++j) {
        if (!warp_wait(b_sft, (uint32_t)n_s & 1u, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        float s[128];
        {
          uint32_t* u = reinterpret_cast<uint32_t*>(s);
          tmem_ld32(lane_base + s_col, *reinterpret_cast<uint32_t(*)[32]>(u));
          tmem_ld32(lane_base + s_col + 32, *reinterpret_cast<uint32_t(*)[32]>(u + 32));
          tmem_ld32(lane_base + s_col + 64, *reinterpret_cast<uint32_t(*)[32]>(u + 64));
          tmem_ld32(lane_base + s_col + 96, *reinterpret_cast<uint32_t(*)[32]>(u + 96));
          tmem_ld_wait();
        }
        tc_fence_before();
        warp_arrive(b_set);  // this warp is done reading S_t
        ++n_s;
        if (quad == 0 && pend >= 0) {  // the previous item's O store has long finished reading its Q tile
          if (lane == 0) {
            bulk_wait_read<0>();
            for (int i = 0; i < pend_n; ++i) mbar_arrive(b_qe + 8 * pend);
          }
          pend = -1;
        }
        const bool diag = j == qt;
        if (diag) {  // keys after the query are masked
          const int kmax = qi - j * AT_B;  // key offsets > kmax are masked
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > kmax) s[c] = -INFINITY;
        }
        // Lazy rescaling: the running max m (log2 units) only moves when the tile's row max
        // exceeds it by more than 8, so p <= 2^8 stays exact in fp32 and bf16; O and l always
        // share the same m, so the result is unchanged.
        const float tmax = row_max128(s) * p.c2;
        float m_new = m;
        if (j == 0 || tmax > m + 8.0f) m_new = fmaxf(m, tmax);
        const bool rescale = j >= 1 && __any_sync(0xffffffffu, m_new != m);
        const float alpha = j == 0 ? 0.f : ex2(m - m_new);
        const float2 nm = make_float2(-m_new, -m_new);
        uint32_t pk[64];
        float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float2 x = fma2(make_float2(s[2 * c], s[2 * c + 1]), c2, nm);
          const float2 pr = make_float2(ex2(x.x), ex2(x.y));
          acc[c & 1] = add2(acc[c & 1], pr);
          pk[c] = pack_bf16x2(pr.x, pr.y);
        }
        l = l * alpha + ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y));
        m = m_new;
        if (j >= 1) {
          // PV_t(j-1) must be done: it reads the P buffer this tile overwrites, and O is
          // rescaled only once that product is in
          if (!warp_wait(b_pvt, (uint32_t)n_pv & 1u, abort_flag, p.status)) { ok = false; break; }
          ++n_pv;
          tc_fence_after();
          if (rescale) {
            uint32_t o[64];
            tmem_ld32(lane_base + o_col, *reinterpret_cast<uint32_t(*)[32]>(o));
            tmem_ld32(lane_base + o_col + 32, *reinterpret_cast<uint32_t(*)[32]>(o + 32));
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 64; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st32(lane_base + o_col, *reinterpret_cast<uint32_t(*)[32]>(o));
            tmem_st32(lane_base + o_col + 32, *reinterpret_cast<uint32_t(*)[32]>(o + 32));
          }
        }
        // P (bf16 pairs) into TMEM: row r, 128 keys = 64 columns
        tmem_st32(lane_base + p_col, *reinterpret_cast<uint32_t(*)[32]>(pk));
        tmem_st32(lane_base + p_col + 32, *reinterpret_cast<uint32_t(*)[32]>(pk + 32));
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(b_pft);
      }
      if (!ok) break;
      // epilogue of this tile: its last PV is done
      if (!warp_wait(b_pvt, (uint32_t)n_pv & 1u, abort_flag, p.status)) break;
      ++n_pv;
      tc_fence_after();
      uint32_t o[64];
      tmem_ld32(lane_base + o_col, *reinterpret_cast<uint32_t(*)[32]>(o));
      tmem_ld32(lane_base + o_col + 32, *reinterpret_cast<uint32_t(*)[32]>(o + 32));
      tmem_ld_wait();
      tc_fence_before();  // the next item's first PV overwrites O after this read
      // O / l rows go into this tile's Q tile, which no product reads any more (the tile's
      // last S completed before it was read); one thread writes the tile out with a tensor
      // store (rows past T are not written)
      const float inv = 1.0f / l;
      const uint32_t ost = sbase + FW_Q + (2 * qs + t) * AT_TILE;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint4 u;
        u.x = pack_bf16x2(__uint_as_float(o[8 * q]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
        u.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
        u.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
        u.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
        st_swizzled(ost, r, q, u);
      }
      fence_async_smem();
      warp_arrive(b_stg + 8 * t);
      if (qi < a.T) a.lse[(long long)bh * a.T + qi] = (m + __log2f(l)) * 0.6931471805599453f;
      if (quad == 0) {
        if (!warp_wait(b_stg + 8 * t, (uint32_t)n_it & 1u, abort_flag, p.status)) break;
        if (lane == 0) {
          if (p.swap_o) tma_store_4d(&tmO, ost, 0, h, qt * AT_B, b);
          else tma_store_4d(&tmO, ost, 0, qt * AT_B, h, b);
          bulk_commit();
        }
        pend = qs;
        pend_n = has1 ? 1 : 2;
      }
      ++n_it;
    }
    if (quad == 0 && lane == 0 && pend >= 0) bulk_wait_all();  // the last item's store is out
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, AT_TMEM_COLS);
  }
}

// ================================================================== backward
// dS = P o (dP - D) with P = 2^(s*scale*log2e - lse*log2e) (the forward's lse),
// dP = dO V^T, D = rowsum(dO o O); dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO.
// Two persistent kernels, both deterministic (no atomics): one owns 128-query
// tiles and accumulates dQ over their key tiles, the other owns 128-key tiles
// and accumulates dK and dV over their query tiles.

constexpr int BW_THREADS = 384;
// warps 0-3: TMA producer, two MMA issuers, one idle; warps 4-11: compute.  Registers:
// 384 x 168 at launch = 64512; the control warpgroup keeps 96, the compute warpgroups take 200
constexpr int BW_REGS_LAUNCH = 168, BW_REGS_CTRL = 96, BW_REGS_COMPUTE = 200;
static_assert(128 * BW_REGS_CTRL + 256 * BW_REGS_COMPUTE <= BW_THREADS * BW_REGS_LAUNCH,
              "the register split must fit in the launch's registers");

struct BwParams {
  AttnArgs a;
  int nq;
  int swap_q, swap_o;  // index order of the q/k/v and the o/dO tensor maps
  float c2;            // scale * log2(e)
  uint32_t idesc_s, idesc_d;  // M128 N128 (K-major B) and M128 N64 (MN-major B)
  unsigned* status;
  int poison;  // test hook (POISON_ATTN_DQ / POISON_ATTN_DKDV): a producer skips its first stage
};

// Column sums of a 32-row x 32-column block held one row per lane: five
// exchange-and-halve shuffle stages leave lane l with column l summed over the
// 32 rows, in a fixed order.
__device__ __forceinline__ float colsum_32x32(const float* v, int lane) {
  float a[16], b[8], c[4], d[2];
  const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4, h2 = lane & 2, h1 = lane & 1;
#pragma unroll
  for (int j = 0; j < 16; ++j) a[j] = (h16 ? v[j + 16] : v[j]) + __shfl_xor_sync(0xffffffffu, h16 ? v[j] : v[j + 16], 16);
#pragma unroll
  for (int j = 0; j < 8; ++j) b[j] = (h8 ? a[j + 8] : a[j]) + __shfl_xor_sync(0xffffffffu, h8 ? a[j] : a[j + 8], 8);
#pragma unroll
  for (int j = 0; j < 4; ++j) c[j] = (h4 ? b[j + 4] : b[j]) + __shfl_xor_sync(0xffffffffu, h4 ? b[j] : b[j + 4], 4);
#pragma unroll
  for (int j = 0; j < 2; ++j) d[j] = (h2 ? c[j + 2] : c[j]) + __shfl_xor_sync(0xffffffffu, h2 ? c[j] : c[j + 2], 2);
  return (h1 ? d[1] : d[0]) + __shfl_xor_sync(0xffffffffu, h1 ? d[0] : d[1], 1);
}

__device__ __forceinline__ void bw_load(const CUtensorMap* tm, int swap, uint32_t dst, uint32_t bar,
                                        int t0, int h, int b) {
  if (swap) tma_load_4d(dst, tm, bar, 0, h, t0, b);
  else tma_load_4d(dst, tm, bar, 0, t0, h, b);
}
// One [128 rows x 64] bf16 tile from shared memory (128B swizzle) to rows t0.. of head (b, h);
// rows past T are not written.
__device__ __forceinline__ void bw_store(const CUtensorMap* tm, int swap, uint32_t src, int t0, int h, int b) {
  if (swap) tma_store_4d(tm, src, 0, h, t0, b);
  else tma_store_4d(tm, src, 0, t0, h, b);
}

// ------------------------------------------------------------------ dQ
// smem: two sets of Q | dO | O (items alternate, so the next item's tiles load while this one
// finishes; a set's Q tile then stages the item's dQ for its tensor store) | K,V ring
// (4 stages); TMEM: S | dP | dQ | dS double buffer.
// The compute warps also form D = rowsum(dO * O) for their query rows from the
// dO and O tiles and store it for the dK/dV kernel, which runs after this one.
constexpr int DQ_STAGES = 4;
constexpr int DQ_Q = 0, DQ_DO = AT_TILE, DQ_O = 2 * AT_TILE, DQ_KV = 6 * AT_TILE;  // set s: + 3 s TILE
constexpr int DQ_BAR = DQ_KV + 2 * DQ_STAGES * AT_TILE;
constexpr int DQ_NBARS = 20;
constexpr int DQ_SMEM = 1024 + DQ_BAR + 8 * (DQ_NBARS + 2);

__global__ void __launch_bounds__(BW_THREADS, 1)
    k_attn_bwd_dq_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                 const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmdQ,
                 const BwParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + DQ_BAR);
  // q_full[2], q_empty[2] (per Q/dO/O set), kv_full[4], kv_empty[4], sdp_full, sdp_empty, ds_full[2],
  // dq_done[2], done (ds_full / dq_done per dS buffer: tile parity)
  const uint32_t b_qf = smem_u32(bars), b_qe = b_qf + 16, b_kvf = b_qe + 16, b_kve = b_kvf + 8 * DQ_STAGES;
  const uint32_t b_sf = b_kve + 8 * DQ_STAGES, b_se = b_sf + 8, b_dsf = b_se + 8, b_dq = b_dsf + 16;
  const uint32_t b_done = b_dq + 16, b_stg = b_done + 8;  // staged: the item's dQ rows are in shared memory
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + DQ_NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + DQ_NBARS + 1);
  const AttnArgs& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BH = a.B * a.H, nitems = p.nq * BH;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_qf + 8 * i, 1);
      // the S / dP issuer's commit after the item's last S / dP, the 8 compute warps (D
      // formed) and the thread whose tensor store of the item's dQ has read the Q tile
      mbar_init(b_qe + 8 * i, 10);
    }
    for (int i = 0; i < DQ_STAGES; ++i) {
      mbar_init(b_kvf + 8 * i, 1);
      mbar_init(b_kve + 8 * i, 1);
    }
    mbar_init(b_sf, 1);
    mbar_init(b_se, 8);  // one arrival per compute warp
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_dsf + 8 * i, 8);
      mbar_init(b_dq + 8 * i, 1);
    }
    mbar_init(b_done, 2);  // one commit per issuer
    mbar_init(b_stg, 8);   // one arrival per compute warp
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  pdl_wait();  // the predecessor kernel is complete: global memory and TMEM are ours
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), AT_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  constexpr uint32_t C_S = 0, C_DP = 128, C_DQ = 256, C_DS = 320;  // dS buffer b at C_DS + 64 b

  if (warp < 4) {
    regs_lower<BW_REGS_CTRL>();
    if (warp == 0) {
      if (lane == 0) {
        int last_par[DQ_STAGES] = {-1, -1, -1, -1}, q_par[2] = {-1, -1}, g = 0;
        bool ok = true;
        for (int w = blockIdx.x, it = 0; ok && w < nitems; w += gridDim.x, ++it) {
          const int qt = p.nq - 1 - w / BH, bh = w % BH, b = bh / a.H, h = bh % a.H;
          const int qs = it & 1;
          const uint32_t qb = sbase + 3 * qs * AT_TILE;
          // set qs was last read by item it - 2
          if (it >= 2 && !mbar_wait(b_qe + 8 * qs, (uint32_t)((it - 2) >> 1) & 1u, abort_flag, p.status)) break;
          mbar_expect_tx(b_qf + 8 * qs, 3 * AT_TILE);
          bw_load(&tmQ, p.swap_q, qb + DQ_Q, b_qf + 8 * qs, qt * AT_B, h, b);
          bw_load(&tmdO, p.swap_o, qb + DQ_DO, b_qf + 8 * qs, qt * AT_B, h, b);
          bw_load(&tmO, p.swap_o, qb + DQ_O, b_qf + 8 * qs, qt * AT_B, h, b);
          q_par[qs] = (it >> 1) & 1;
          for (int j = 0; j <= qt; ++j, ++g) {
            const int st = g % DQ_STAGES;
            const uint32_t ph = (uint32_t)(g / DQ_STAGES) & 1u;
            if (!mbar_wait(b_kve + 8 * st, ph ^ 1u, abort_flag, p.status)) { ok = false; break; }
            if ((p.poison & POISON_ATTN_DQ) && g == 0) continue;
            const uint32_t kd = sbase + DQ_KV + st * 2 * AT_TILE;
            mbar_expect_tx(b_kvf + 8 * st, 2 * AT_TILE);
            bw_load(&tmK, p.swap_q, kd, b_kvf + 8 * st, j * AT_B, h, b);
            bw_load(&tmV, p.swap_q, kd + AT_TILE, b_kvf + 8 * st, j * AT_B, h, b);
            last_par[st] = (int)ph;
          }
        }
        for (int i = 0; i < 2; ++i)
          if (q_par[i] >= 0) mbar_wait_drain(b_qf + 8 * i, (uint32_t)q_par[i]);
        for (int i = 0; i < DQ_STAGES; ++i)
          if (last_par[i] >= 0) mbar_wait_drain(b_kvf + 8 * i, (uint32_t)last_par[i]);
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // ---------------- S / dP issuer: S(g) = Q K_j^T and dP(g) = dO V_j^T once K_j, V_j
        // have landed and the compute warps have read S(g-1), dP(g-1)
        bool ok = true;
        int g = 0;
        for (int w = blockIdx.x, it = 0; ok && w < nitems; w += gridDim.x, ++it) {
          const int nk = p.nq - w / BH;
          const int qs = it & 1;
          const uint32_t qb = sbase + 3 * qs * AT_TILE;
          if (!mbar_wait(b_qf + 8 * qs, (uint32_t)(it >> 1) & 1u, abort_flag, p.status)) break;
          for (int j = 0; j < nk; ++j, ++g) {
            const int st = g % DQ_STAGES;
            if (!mbar_wait(b_kvf + 8 * st, (uint32_t)(g / DQ_STAGES) & 1u, abort_flag, p.status)) {
              ok = false;
              break;
            }
            if (g >= 1 && !mbar_wait(b_se, (uint32_t)(g - 1) & 1u, abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint32_t kd = sbase + DQ_KV + st * 2 * AT_TILE;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16(tmem + C_S, operand_desc(qb + DQ_Q, 0, k), operand_desc(kd, 0, k), p.idesc_s, k > 0 ? 1u : 0u);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16(tmem + C_DP, operand_desc(qb + DQ_DO, 0, k), operand_desc(kd + AT_TILE, 0, k), p.idesc_s,
                       k > 0 ? 1u : 0u);
            mma_commit(b_sf);
            if (j == nk - 1) mma_commit(b_qe + 8 * qs);
          }
        }
        mma_commit(b_done);
        mbar_wait_drain(b_done, 0);
      }
    } else if (warp == 2) {
      if (lane == 0) {
        // ---------------- dQ issuer: dQ += dS(g) K_j once the compute warps have written
        // dS(g); its commit also frees K_j / V_j (S(g) and dP(g), the stage's other
        // readers, were complete before dS(g) could be formed)
        bool ok = true;
        int g = 0;
        for (int w = blockIdx.x; ok && w < nitems; w += gridDim.x) {
          const int nk = p.nq - w / BH;
          for (int j = 0; j < nk; ++j, ++g) {
            const int db = g & 1;
            if (!mbar_wait(b_dsf + 8 * db, (uint32_t)(g >> 1) & 1u, abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint32_t kd = sbase + DQ_KV + (g % DQ_STAGES) * 2 * AT_TILE;
            // A = dS in TMEM: 16 keys per MMA = 8 columns of bf16 pairs
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_bf16_tmem_a(tmem + C_DQ, tmem + C_DS + db * 64 + kk * 8, operand_desc(kd, 1, kk), p.idesc_d,
                              (j > 0 || kk > 0) ? 1u : 0u);
            mma_commit(b_dq + 8 * db);
            mma_commit(b_kve + 8 * (g % DQ_STAGES));
          }
        }
        mma_commit(b_done);
        mbar_wait_drain(b_done, 0);
      }
    }
  } else {
    regs_raise<BW_REGS_COMPUTE>();
    const int quad = warp & 3, half = (warp - 4) >> 2;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    bool ok = true;
    int g = 0;
    int pend = -1;  // warp 4: the Q set whose dQ tensor store is in flight
    for (int w = blockIdx.x, it = 0; ok && w < nitems; w += gridDim.x, ++it) {
      const int qt = p.nq - 1 - w / BH, bh = w % BH, b = bh / a.H, h = bh % a.H;
      const int nk = qt + 1;
      const int qi = qt * AT_B + r;
      const bool valid = qi < a.T;
      const float lse2 = valid ? a.lse[(long long)bh * a.T + qi] * 1.4426950408889634f : 0.f;
      // D = sum over d of dO[q, d] O[q, d] from the staged tiles (row r: 128 B, 16-byte
      // piece c at ((c ^ (r & 7)) << 4), the 128B swizzle), pieces in order
      const int qs = it & 1;
      const uint32_t qb = sbase + 3 * qs * AT_TILE;
      if (!warp_wait(b_qf + 8 * qs, (uint32_t)(it >> 1) & 1u, abort_flag, p.status)) break;
      float Dr = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t off = (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
        uint32_t x[4], y[4];
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3])
                     : "r"(qb + DQ_DO + off));
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(y[0]), "=r"(y[1]), "=r"(y[2]), "=r"(y[3])
                     : "r"(qb + DQ_O + off));
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          Dr = fmaf(__uint_as_float(x[e] << 16), __uint_as_float(y[e] << 16), Dr);
          Dr = fmaf(__uint_as_float(x[e] & 0xFFFF0000u), __uint_as_float(y[e] & 0xFFFF0000u), Dr);
        }
      }
      if (!valid) Dr = 0.f;
      if (valid && half == 0) a.Dbuf[(long long)bh * a.T + qi] = Dr;
      warp_arrive(b_qe + 8 * qs);  // this warp is done with the item's dO and O tiles
      for (int j = 0; j < nk; ++j, ++g) {
        if (!warp_wait(b_sf, (uint32_t)g & 1u, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[64], dv[64];
        tmem_ld32(lane_base + C_S + half * 64, *reinterpret_cast<uint32_t(*)[32]>(sv));
        tmem_ld32(lane_base + C_S + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
        tmem_ld32(lane_base + C_DP + half * 64, *reinterpret_cast<uint32_t(*)[32]>(dv));
        tmem_ld32(lane_base + C_DP + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(dv + 32));
        tmem_ld_wait();
        tc_fence_before();
        warp_arrive(b_se);
        if (warp == 4 && pend >= 0) {  // the previous item's dQ store has long finished reading its Q tile
          if (lane == 0) {
            bulk_wait_read<0>();
            mbar_arrive(b_qe + 8 * pend);
          }
          pend = -1;
        }
        const int kmask = j == qt ? qi - j * AT_B - half * 64 : AT_B;  // key offsets > kmask are masked
        const float2 c2 = make_float2(p.c2, p.c2), nl = make_float2(-lse2, -lse2);
        const float2 nd = make_float2(-Dr, -Dr);
        uint32_t pk[32];
        // dS = P (dP - D) for a pair of key columns
        auto pair = [&](int c, bool zero0, bool zero1) {
          const float2 x = fma2(make_float2(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1])), c2, nl);
          float2 pr = make_float2(ex2(x.x), ex2(x.y));
          if (zero0) pr.x = 0.f;
          if (zero1) pr.y = 0.f;
          const float2 t = mul2(pr, add2(make_float2(__uint_as_float(dv[2 * c]), __uint_as_float(dv[2 * c + 1])), nd));
          pk[c] = pack_bf16x2(t.x, t.y);
        };
        if (j == qt) {  // diagonal tile: keys after the query are masked
#pragma unroll
          for (int c = 0; c < 32; ++c) pair(c, 2 * c > kmask, 2 * c + 1 > kmask);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) pair(c, false, false);
        }
        // this dS buffer is free once the dQ MMA of tile g-2 has completed
        const int db = g & 1;
        if (g >= 2 && !warp_wait(b_dq + 8 * db, (uint32_t)((g - 2) >> 1) & 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tmem_st32(lane_base + C_DS + db * 64 + half * 32, pk);
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(b_dsf + 8 * db);
      }
      if (!ok) break;
      if (!warp_wait(b_dq + 8 * ((g - 1) & 1), (uint32_t)((g - 1) >> 1) & 1u, abort_flag, p.status)) break;
      tc_fence_after();
      uint32_t o[32];
      tmem_ld32(lane_base + C_DQ + half * 32, o);
      tmem_ld_wait();
      tc_fence_before();
      if (a.bias_part) {  // this warp's 32 rows x 32 dq columns, summed per column
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = valid ? __uint_as_float(o[i]) * a.scale : 0.f;
        const float cs = colsum_32x32(v, lane);
        const long long prow = ((long long)b * p.nq + qt) * 4 + quad;
        a.bias_part[prow * 3 * a.H * AT_D + h * AT_D + half * 32 + lane] = cs;
      }
      // dQ rows go into the item's Q tile, which no product reads any more (the item's last
      // S completed before its last dS was formed); one thread writes the tile out with a
      // tensor store (rows past T are not written).
      const uint32_t qst = qb + DQ_Q;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 u;
        u.x = pack_bf16x2(__uint_as_float(o[8 * q]) * a.scale, __uint_as_float(o[8 * q + 1]) * a.scale);
        u.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * a.scale, __uint_as_float(o[8 * q + 3]) * a.scale);
        u.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * a.scale, __uint_as_float(o[8 * q + 5]) * a.scale);
        u.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * a.scale, __uint_as_float(o[8 * q + 7]) * a.scale);
        st_swizzled(qst, r, half * 4 + q, u);
      }
      fence_async_smem();
      warp_arrive(b_stg);
      if (warp == 4) {
        if (!warp_wait(b_stg, (uint32_t)it & 1u, abort_flag, p.status)) break;
        if (lane == 0) {
          bw_store(&tmdQ, p.swap_q, qst, qt * AT_B, h, b);
          bulk_commit();
        }
        pend = qs;
      }
    }
    if (warp == 4 && lane == 0 && pend >= 0) bulk_wait_all();  // the last item's store is out
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, AT_TMEM_COLS);
  }
}

// ------------------------------------------------------------------ dK, dV
// smem: two sets of K | V (items alternate, so the next item's K and V load while this
// one finishes; a set then stages the item's dK | dV for the tensor stores) | Q,dO ring
// (4 stages) | lse2, D ring (4 x 1 KB);
// TMEM: S^T | dP^T | dV | dK | P^T | dS^T
constexpr int DK_STAGES = 4;
constexpr int DK_K = 0, DK_V = AT_TILE, DK_QD = 4 * AT_TILE, DK_LD = DK_QD + 2 * DK_STAGES * AT_TILE;  // set s: K, V at + 2 s TILE
constexpr int DK_BAR = DK_LD + DK_STAGES * 1024;
constexpr int DK_NBARS = 20;
constexpr int DK_SMEM = 1024 + DK_BAR + 8 * (DK_NBARS + 2);

__global__ void __launch_bounds__(BW_THREADS, 1)
    k_attn_bwd_dkdv_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                       const BwParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  // stage s: for each query pair (2i, 2i+1) the float4 {-lse2[2i], -lse2[2i+1], -D[2i], -D[2i+1]}
  float* ldbuf = reinterpret_cast<float*>(smem + DK_LD);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + DK_BAR);
  // kv_full[2], kv_empty[2] (per K/V set), qd_full[4], qd_empty[4], sdp_full, sdp_empty, ds_full,
  // mma_done, done, staged (the item's dK / dV rows are in shared memory)
  const uint32_t b_kvf = smem_u32(bars), b_kve = b_kvf + 16, b_qdf = b_kve + 16, b_qde = b_qdf + 8 * DK_STAGES;
  const uint32_t b_sf = b_qde + 8 * DK_STAGES, b_se = b_sf + 8, b_dsf = b_se + 8, b_mm = b_dsf + 8;
  const uint32_t b_done = b_mm + 8, b_stg = b_done + 8;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + DK_NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + DK_NBARS + 1);
  const AttnArgs& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BH = a.B * a.H, nitems = p.nq * BH;
  // work item w: key tile w / BH (tile 0 has the most query tiles), (batch, head) = w % BH

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_kvf + 8 * i, 1);
      mbar_init(b_kve + 8 * i, 1);  // the epilogue's tensor stores have read the set (it stages dK, dV)
    }
    for (int i = 0; i < DK_STAGES; ++i) {
      mbar_init(b_qdf + 8 * i, 2);  // the TMA expect_tx arrive + the warp that staged lse2 / D
      mbar_init(b_qde + 8 * i, 1);
    }
    mbar_init(b_sf, 1);
    mbar_init(b_se, 8);  // one arrival per compute warp
    mbar_init(b_dsf, 8);
    mbar_init(b_mm, 1);
    mbar_init(b_done, 2);  // one commit per issuer
    mbar_init(b_stg, 8);   // one arrival per compute warp
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  pdl_wait();  // the predecessor kernel is complete: global memory and TMEM are ours
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), AT_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  constexpr uint32_t C_S = 0, C_DP = 128, C_DV = 256, C_DK = 320, C_PT = 384, C_DST = 448;

  if (warp < 4) {
    regs_lower<BW_REGS_CTRL>();
    if (warp == 0) {
      // ---------------- producer warp: TMA by lane 0, lse2 / D staged by all lanes
      // Each lane's four lse and D values for a query tile are loaded one tile ahead, so
      // their global-memory latency overlaps the wait for the ring stage.
      int last_par[DK_STAGES] = {-1, -1, -1, -1}, kv_par[2] = {-1, -1}, g = 0;
      bool ok = true;
      float nl[4], nd[4];  // lse and D of the next query tile to stage (this lane's 4 queries)
      auto fetch = [&](int bh, int i) {
  #pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int q = i * AT_B + lane * 4 + e;
          const bool v = q < a.T;
          nl[e] = v ? a.lse[(long long)bh * a.T + q] : INFINITY;
          nd[e] = v ? a.Dbuf[(long long)bh * a.T + q] : 0.f;
        }
      };
      if (blockIdx.x < nitems) fetch(blockIdx.x % BH, blockIdx.x / BH);
      for (int w = blockIdx.x, it = 0; ok && w < nitems; w += gridDim.x, ++it) {
        const int kt = w / BH, bh = w % BH, b = bh / a.H, h = bh % a.H;
        const int ks = it & 1;  // K/V set of this item
        if (it >= 2 && !warp_wait(b_kve + 8 * ks, (uint32_t)((it - 2) >> 1) & 1u, abort_flag, p.status)) break;
        if (lane == 0) {
          mbar_expect_tx(b_kvf + 8 * ks, 2 * AT_TILE);
          bw_load(&tmK, p.swap_q, sbase + DK_K + 2 * ks * AT_TILE, b_kvf + 8 * ks, kt * AT_B, h, b);
          bw_load(&tmV, p.swap_q, sbase + DK_V + 2 * ks * AT_TILE, b_kvf + 8 * ks, kt * AT_B, h, b);
        }
        kv_par[ks] = (it >> 1) & 1;
        for (int i = kt; i < p.nq; ++i, ++g) {
          const int st = g % DK_STAGES;
          const uint32_t ph = (uint32_t)(g / DK_STAGES) & 1u;
          if (!warp_wait(b_qde + 8 * st, ph ^ 1u, abort_flag, p.status)) { ok = false; break; }
          if (lane == 0 && !((p.poison & POISON_ATTN_DKDV) && g == 0)) {
            const uint32_t qd = sbase + DK_QD + st * 2 * AT_TILE;
            mbar_expect_tx(b_qdf + 8 * st, 2 * AT_TILE);
            bw_load(&tmQ, p.swap_q, qd, b_qdf + 8 * st, i * AT_B, h, b);
            bw_load(&tmdO, p.swap_o, qd + AT_TILE, b_qdf + 8 * st, i * AT_B, h, b);
          }
          float* lb = ldbuf + st * 256;
  #pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = lane * 4 + e;
            const int slot = (c >> 1) * 4 + (c & 1);
            lb[slot] = -nl[e] * 1.4426950408889634f;  // rows past T: -inf, so P = 0 there
            lb[slot + 2] = -nd[e];
          }
          warp_arrive(b_qdf + 8 * st);
          if (!((p.poison & POISON_ATTN_DKDV) && g == 0)) last_par[st] = (int)ph;
          // the next tile's values: this item's next query tile, or the next item's first
          if (i + 1 < p.nq) fetch(bh, i + 1);
          else if (w + (int)gridDim.x < nitems) fetch((w + gridDim.x) % BH, (w + gridDim.x) / BH);
        }
      }
      if (lane == 0) {
        for (int i = 0; i < 2; ++i)
          if (kv_par[i] >= 0) mbar_wait_drain(b_kvf + 8 * i, (uint32_t)kv_par[i]);
        for (int i = 0; i < DK_STAGES; ++i)
          if (last_par[i] >= 0) mbar_wait_drain(b_qdf + 8 * i, (uint32_t)last_par[i]);
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // ---------------- S^T / dP^T issuer: S^T(g) = K Q_i^T and dP^T(g) = V dO_i^T once
        // Q_i, dO_i have landed and the compute warps have read S^T(g-1), dP^T(g-1)
        bool ok = true;
        int g = 0;
        for (int w = blockIdx.x, it = 0; ok && w < nitems; w += gridDim.x, ++it) {
          const int n = p.nq - w / BH;  // query tiles kt .. nq-1
          const int ks = it & 1;
          const uint32_t kd = sbase + DK_K + 2 * ks * AT_TILE, vd = sbase + DK_V + 2 * ks * AT_TILE;
          if (!mbar_wait(b_kvf + 8 * ks, (uint32_t)(it >> 1) & 1u, abort_flag, p.status)) break;
          for (int j = 0; j < n; ++j, ++g) {
            const int st = g % DK_STAGES;
            if (!mbar_wait(b_qdf + 8 * st, (uint32_t)(g / DK_STAGES) & 1u, abort_flag, p.status)) {
              ok = false;
              break;
            }
            if (g >= 1 && !mbar_wait(b_se, (uint32_t)(g - 1) & 1u, abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint32_t qd = sbase + DK_QD + st * 2 * AT_TILE;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16(tmem + C_S, operand_desc(kd, 0, k), operand_desc(qd, 0, k), p.idesc_s, k > 0 ? 1u : 0u);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16(tmem + C_DP, operand_desc(vd, 0, k), operand_desc(qd + AT_TILE, 0, k), p.idesc_s,
                       k > 0 ? 1u : 0u);
            mma_commit(b_sf);
          }
        }
        mma_commit(b_done);
        mbar_wait_drain(b_done, 0);
      }
    } else if (warp == 2) {
      if (lane == 0) {
        // ---------------- dV / dK issuer: dV += P^T(g) dO_i, dK += dS^T(g) Q_i once the
        // compute warps have written P^T(g), dS^T(g).  Its commit frees the Q_i / dO_i stage
        // (the S^T and dP^T products, its other readers, were complete before dS^T could be
        // formed).
        bool ok = true;
        int g = 0;
        for (int w = blockIdx.x; ok && w < nitems; w += gridDim.x) {
        const int n = p.nq - w / BH;
        for (int j = 0; j < n; ++j, ++g) {
        if (!mbar_wait(b_dsf, (uint32_t)g & 1u, abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint32_t qd = sbase + DK_QD + (g % DK_STAGES) * 2 * AT_TILE;
            // A = P^T / dS^T in TMEM: 16 queries per MMA = 8 columns of bf16 pairs
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_bf16_tmem_a(tmem + C_DV, tmem + C_PT + kk * 8, operand_desc(qd + AT_TILE, 1, kk), p.idesc_d,
                              (j > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_bf16_tmem_a(tmem + C_DK, tmem + C_DST + kk * 8, operand_desc(qd, 1, kk), p.idesc_d,
                              (j > 0 || kk > 0) ? 1u : 0u);
            mma_commit(b_mm);
            mma_commit(b_qde + 8 * (g % DK_STAGES));
            }
            }
        mma_commit(b_done);
        mbar_wait_drain(b_done, 0);
      }
    }
  } else {
    regs_raise<BW_REGS_COMPUTE>();
    const int quad = warp & 3, half = (warp - 4) >> 2;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    bool ok = true;
    int g = 0;
    int pend = -1;  // warp 4: the K/V set whose tensor stores are in flight
    for (int w = blockIdx.x, it = 0; ok && w < nitems; w += gridDim.x, ++it) {
      const int kt = w / BH, bh = w % BH, b = bh / a.H, h = bh % a.H;
      const int kr = kt * AT_B + r;
      for (int i = kt; i < p.nq; ++i, ++g) {
        const int st = g % DK_STAGES;
        // lse2 / D of this query tile (staged with the Q / dO tiles)
        if (!warp_wait(b_qdf + 8 * st, (uint32_t)(g / DK_STAGES) & 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        if (!warp_wait(b_sf, (uint32_t)g & 1u, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[64], dv[64];
        tmem_ld32(lane_base + C_S + half * 64, *reinterpret_cast<uint32_t(*)[32]>(sv));
        tmem_ld32(lane_base + C_S + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
        tmem_ld32(lane_base + C_DP + half * 64, *reinterpret_cast<uint32_t(*)[32]>(dv));
        tmem_ld32(lane_base + C_DP + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(dv + 32));
        tmem_ld_wait();
        tc_fence_before();
        warp_arrive(b_se);
        if (warp == 4 && pend >= 0) {  // the previous item's stores have long finished reading its set
          if (lane == 0) {
            bulk_wait_read<0>();
            mbar_arrive(b_kve + 8 * pend);
          }
          pend = -1;
        }
        const float4* ld4 = reinterpret_cast<const float4*>(ldbuf + st * 256) + half * 32;
        const float2 c2 = make_float2(p.c2, p.c2);
        uint32_t pp[32], pd[32];
        // P^T = 2^(s c2 - lse2) and dS^T = P^T (dP^T - D) for a pair of query columns
        auto pair = [&](int c, bool zero0, bool zero1) {
          const float4 w = ld4[c];  // -lse2[q], -lse2[q+1], -D[q], -D[q+1]
          const float2 x = fma2(make_float2(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1])), c2,
                                make_float2(w.x, w.y));
          float2 pr = make_float2(ex2(x.x), ex2(x.y));
          if (zero0) pr.x = 0.f;
          if (zero1) pr.y = 0.f;
          pp[c] = pack_bf16x2(pr.x, pr.y);
          const float2 t = mul2(pr, add2(make_float2(__uint_as_float(dv[2 * c]), __uint_as_float(dv[2 * c + 1])),
                                         make_float2(w.z, w.w)));
          pd[c] = pack_bf16x2(t.x, t.y);
        };
        if (i == kt) {  // diagonal tile: queries before this key (offsets below kmask) are masked
          const int kmask = r - half * 64;
#pragma unroll
          for (int c = 0; c < 32; ++c) pair(c, 2 * c < kmask, 2 * c + 1 < kmask);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) pair(c, false, false);
        }
        // P^T / dS^T are free once the previous dV / dK MMAs have completed
        if (g >= 1 && !warp_wait(b_mm, (uint32_t)(g - 1) & 1u, abort_flag, p.status)) { ok = false; break; }
        tmem_st32(lane_base + C_PT + half * 32, pp);
        tmem_st32(lane_base + C_DST + half * 32, pd);
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(b_dsf);
      }
      if (!ok) break;
      if (!warp_wait(b_mm, (uint32_t)(g - 1) & 1u, abort_flag, p.status)) break;
      tc_fence_after();
      uint32_t ov[32], ok_[32];
      tmem_ld32(lane_base + C_DV + half * 32, ov);
      tmem_ld32(lane_base + C_DK + half * 32, ok_);
      tmem_ld_wait();
      tc_fence_before();
      if (a.bias_part) {  // this warp's 32 key rows x 32 columns of dk and of dv, summed per column
        const int C = a.H * AT_D;
        const long long prow = ((long long)b * p.nq + kt) * 4 + quad;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = kr < a.T ? __uint_as_float(ok_[i]) * a.scale : 0.f;
        float cs = colsum_32x32(v, lane);
        a.bias_part[prow * 3 * C + C + h * AT_D + half * 32 + lane] = cs;
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = kr < a.T ? __uint_as_float(ov[i]) : 0.f;
        cs = colsum_32x32(v, lane);
        a.bias_part[prow * 3 * C + 2 * C + h * AT_D + half * 32 + lane] = cs;
      }
      // dK (scaled) and dV rows go into the item's K / V tiles, which no product reads any
      // more (the item's last S^T / dP^T completed before its last dS^T was formed); one
      // thread writes both tiles out with tensor stores (rows past T are not written), and
      // the set goes back to the producer once those stores have read it.
      const int ks = it & 1;
      const uint32_t kst = sbase + DK_K + 2 * ks * AT_TILE, vst = sbase + DK_V + 2 * ks * AT_TILE;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 u, k;
        u.x = pack_bf16x2(__uint_as_float(ov[8 * q]), __uint_as_float(ov[8 * q + 1]));
        u.y = pack_bf16x2(__uint_as_float(ov[8 * q + 2]), __uint_as_float(ov[8 * q + 3]));
        u.z = pack_bf16x2(__uint_as_float(ov[8 * q + 4]), __uint_as_float(ov[8 * q + 5]));
        u.w = pack_bf16x2(__uint_as_float(ov[8 * q + 6]), __uint_as_float(ov[8 * q + 7]));
        k.x = pack_bf16x2(__uint_as_float(ok_[8 * q]) * a.scale, __uint_as_float(ok_[8 * q + 1]) * a.scale);
        k.y = pack_bf16x2(__uint_as_float(ok_[8 * q + 2]) * a.scale, __uint_as_float(ok_[8 * q + 3]) * a.scale);
        k.z = pack_bf16x2(__uint_as_float(ok_[8 * q + 4]) * a.scale, __uint_as_float(ok_[8 * q + 5]) * a.scale);
        k.w = pack_bf16x2(__uint_as_float(ok_[8 * q + 6]) * a.scale, __uint_as_float(ok_[8 * q + 7]) * a.scale);
        st_swizzled(vst, r, half * 4 + q, u);
        st_swizzled(kst, r, half * 4 + q, k);
      }
      fence_async_smem();
      warp_arrive(b_stg);
      if (warp == 4) {
        if (!warp_wait(b_stg, (uint32_t)it & 1u, abort_flag, p.status)) break;
        if (lane == 0) {
          bw_store(&tmdK, p.swap_q, kst, kt * AT_B, h, b);
          bw_store(&tmdV, p.swap_q, vst, kt * AT_B, h, b);
          bulk_commit();
        }
        pend = ks;
      }
    }
    if (warp == 4 && lane == 0 && pend >= 0) bulk_wait_all();  // the last item's stores are out
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, AT_TMEM_COLS);
  }
}

typedef CUresult (*PFN_encodeTiled_t)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                      const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                      const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                      CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

PFN_encodeTiled_t encode_fn() {
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

// 4-D map over a strided [B, H, T, 64] bf16 view: dims (d, t, h, b), or (d, h, t, b)
// when the head stride is the smaller one; boxes of 128 rows x 64 bf16, 128B swizzle.
bool make_head_map(CUtensorMap* tm, const void* base, const AttnArgs& a, int swap) {
  PFN_encodeTiled_t enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4], el[4] = {1, 1, 1, 1};
  dims[0] = AT_D;
  box[0] = AT_D;
  if (swap) {
    dims[1] = a.H; dims[2] = a.T;
    strides[0] = a.sh * 2; strides[1] = a.st * 2;
    box[1] = 1; box[2] = AT_B;
  } else {
    dims[1] = a.T; dims[2] = a.H;
    strides[0] = a.st * 2; strides[1] = a.sh * 2;
    box[1] = AT_B; box[2] = 1;
  }
  dims[3] = a.B;
  strides[2] = a.sb * 2;
  box[3] = 1;
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
                   el, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

uint32_t mma_idesc(int n, int b_mn) {
  // kind::f16: D fp32, A and B bf16, A K-major, B K- or MN-major, N >> 3, M = 128 >> 4
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(AT_B >> 4) << 24);
}

}  // namespace

static bool tc_args_ok(const AttnArgs& a) {
  if (a.d != AT_D || a.T <= 0 || a.B <= 0 || a.H <= 0) return false;
  if (a.st % 8 || a.sh % 8 || a.sb % 8 || a.ost % 8 || a.osh % 8 || a.osb % 8) return false;
  return true;
}

int attn_fwd_tc(const AttnArgs& a, cudaStream_t s) {
  if (!tc_args_ok(a)) return (int)cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(a.q) | reinterpret_cast<uintptr_t>(a.k) |
       reinterpret_cast<uintptr_t>(a.v) | reinterpret_cast<uintptr_t>(a.o)) & 15)
    return (int)cudaErrorInvalidValue;
  static PerDeviceOnce attr;
  cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(k_attn_fwd_tc), AT_SMEM, &attr);
  if (e != cudaSuccess) return (int)e;
  AtParams p;
  p.a = a;
  p.nq = (a.T + AT_B - 1) / AT_B;
  p.nqp = (p.nq + 1) / 2;
  p.swap_ht = a.sh < a.st ? 1 : 0;
  p.swap_o = a.osh < a.ost ? 1 : 0;
  p.c2 = a.scale * 1.4426950408889634f;
  p.idesc_s = mma_idesc(AT_B, 0);
  p.idesc_pv = mma_idesc(AT_D, 1);
  p.status = a.status;
  p.poison = test_poison();
  AttnArgs ao = a;  // o has its own strides
  ao.st = a.ost; ao.sh = a.osh; ao.sb = a.osb;
  CUtensorMap tq, tk, tv, to;
  if (!make_head_map(&tq, a.q, a, p.swap_ht) || !make_head_map(&tk, a.k, a, p.swap_ht) ||
      !make_head_map(&tv, a.v, a, p.swap_ht) || !make_head_map(&to, a.o, ao, p.swap_o))
    return (int)cudaErrorInvalidValue;
  const long long items = (long long)p.nqp * a.B * a.H;
  const int grid = (int)(items < num_sms() ? items : num_sms());
  launch_k(k_attn_fwd_tc, grid, AT_THREADS, AT_SMEM, s, tq, tk, tv, to, p);
  return (int)cudaGetLastError();
}

int attn_bwd_tc(const AttnArgs& a, cudaStream_t s) {
  if (!tc_args_ok(a)) return (int)cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(a.q) | reinterpret_cast<uintptr_t>(a.k) |
       reinterpret_cast<uintptr_t>(a.v) | reinterpret_cast<uintptr_t>(a.dO) |
       reinterpret_cast<uintptr_t>(a.o) | reinterpret_cast<uintptr_t>(a.dq) |
       reinterpret_cast<uintptr_t>(a.dk) | reinterpret_cast<uintptr_t>(a.dv)) & 15 || !a.Dbuf)
    return (int)cudaErrorInvalidValue;
  static PerDeviceOnce attr_dq, attr_dkdv;
  cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(k_attn_bwd_dq_tc), DQ_SMEM, &attr_dq);
  if (e == cudaSuccess)
    e = smem_limit_once(reinterpret_cast<const void*>(k_attn_bwd_dkdv_tc), DK_SMEM, &attr_dkdv);
  if (e != cudaSuccess) return (int)e;
  BwParams p;
  p.a = a;
  p.nq = (a.T + AT_B - 1) / AT_B;
  p.swap_q = a.sh < a.st ? 1 : 0;
  p.swap_o = a.osh < a.ost ? 1 : 0;
  p.c2 = a.scale * 1.4426950408889634f;
  p.idesc_s = mma_idesc(AT_B, 0);
  p.idesc_d = mma_idesc(AT_D, 1);
  p.status = a.status;
  p.poison = test_poison();
  AttnArgs ao = a;  // dO shares the o strides
  ao.st = a.ost; ao.sh = a.osh; ao.sb = a.osb;
  CUtensorMap tq, tk, tv, tdo, to, tdk, tdv, tdq;
  if (!make_head_map(&tq, a.q, a, p.swap_q) || !make_head_map(&tk, a.k, a, p.swap_q) ||
      !make_head_map(&tv, a.v, a, p.swap_q) || !make_head_map(&tdo, a.dO, ao, p.swap_o) ||
      !make_head_map(&to, a.o, ao, p.swap_o) || !make_head_map(&tdk, a.dk, a, p.swap_q) ||
      !make_head_map(&tdv, a.dv, a, p.swap_q) || !make_head_map(&tdq, a.dq, a, p.swap_q))
    return (int)cudaErrorInvalidValue;
  const long long items = (long long)p.nq * a.B * a.H;
  const int grid = (int)(items < num_sms() ? items : num_sms());
  // dQ first: it also writes D = rowsum(dO * O), which the dK/dV kernel reads
  launch_k(k_attn_bwd_dq_tc, grid, BW_THREADS, DQ_SMEM, s, tq, tk, tv, tdo, to, tdq, p);
  launch_k(k_attn_bwd_dkdv_tc, grid, BW_THREADS, DK_SMEM, s, tq, tk, tv, tdo, tdk, tdv, p);
  return (int)cudaGetLastError();
}

}  // namespace gpt2k
