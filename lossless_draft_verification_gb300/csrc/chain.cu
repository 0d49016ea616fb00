// Chain speculative sampling, greedy chain verification and the analytic
// acceptance c*, for sm_103a.
//
// Method (DART reading notes §2.3 eq. (3)-(4); DSpark paper guide, verification
// rule; speculative-decoding survey §1.2-§1.3): accept draft token x_k with
// probability min(1, q_k(x_k)/p_k(x_k)); the first rejection at k discards the
// rest and draws the correction from r = [q_k - p_k]_+ / R; with no rejection
// the bonus token is drawn from q at the next position.  c*_k =
// 1 - 1/2 ||p_k - q_k||_1 = 1 - R_k.
//
// Kernels
//   chain_stats   one thread-block cluster per row pair (target row, draft row)
//                 of one request position; each CTA holds its share of both rows
//                 in registers (8 warps x one warp tile each).  Pass 1: per-tile
//                 max and sum of 2^(x*c2 - m) for q and p.  The cluster combines
//                 the tile partials through distributed shared memory into the
//                 row's (max, normaliser).  Pass 2 (from registers): per-tile
//                 residual mass sum [q - p]_+ and q mass.  CTA rank 0 evaluates
//                 the accept threshold min(1, q(x)/p(x)).  HBM reads each logit
//                 exactly once.
//   chain_finish  one CTA per request: warp ballot over the accept tests ->
//                 first rejection A; c* from the tile partials; inverse-CDF
//                 draw: prefix over tile masses, then one tile rescanned with the
//                 same per-element arithmetic as pass 2.
//   argmax_tiles  per warp tile (max, lowest index); greedy_finish combines
//                 them and walks the chain at T = 0.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "host_common.h"

#include <atomic>

namespace specv {

constexpr int kStatsWarps = 8;        // warps (tiles) per CTA in chain_stats
constexpr int kMaxCluster = 16;
constexpr int kMaxTiles = kStatsWarps * kMaxCluster;   // 128 tiles per row
constexpr int kFinishThreads = 256;
constexpr int kMaxCompactRequests = 4096;   // ragged batches up to this R walk only their live items
constexpr int kArgmaxWarps = 8;

struct RowRec {
  RowStats s;
};

struct StatsArgs {
  const void* target;
  const void* draft;          // null for bonus-only use
  const int32_t* tokens;      // [R, gamma] or null (tv_accept)
  const int32_t* lengths;     // [R] or null
  void* workspace;
  RowRec* rows;               // [R * P]
  TileStats* tiles;           // [R * P, ntile_stride]
  long V;
  int gamma;
  int P;                      // item positions per request (gamma+1 with bonus, gamma without)
  int Pt, Pd;                 // positions per request in target / draft tensors
  int nwt;                    // tiles per row (<= C * kStatsWarps)
  int ntile_stride;
  int with_bonus;
  float c2;                   // log2(e) / T
};

// ---------------------------------------------------------------------------
// Shared-memory layout of the target row's exponentials: for warp w, slot j,
// half h (elements 4h .. 4h+3 of the slot) lane l's float4 sits at
// [(w * VPT + j) * 2 + h][l], so a warp's 128-bit stores and loads are
// contiguous (conflict-free).  Only the 16-byte path keeps them (VW == 8 or 4).
//
// NW warps per CTA (8 or 16).  KEEP_P: the draft row's float32 exponentials stay
// in registers for pass 2; otherwise pass 2 recomputes them from the raw logits
// (fewer registers, so 16-warp CTAs fit two per SM).
template <typename Elem, bool VEC, int VPT, int NW, bool KEEP_P>
__global__ void __launch_bounds__(NW * 32, 2) chain_stats_kernel(StatsArgs a) {
  using S = Slot<Elem, VEC>;
  constexpr int VW = S::VW;
  constexpr int NE = VPT * VW;                 // elements per lane per row
  constexpr int H = VW / 4;                    // float4 per slot (16-byte path)
  extern __shared__ float4 s_exp[];            // target exponentials (16-byte path)
  __shared__ float4 s_warp[NW];
  __shared__ float4 s_cta;

  const uint32_t C = cluster_nctarank();
  const uint32_t rank = cluster_ctarank();
  const int item = blockIdx.x / C;
  const int r = item / a.P;
  const int k = item - r * a.P;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (item == 0 && rank == 0 && threadIdx.x == 0) *reinterpret_cast<int*>(a.workspace) = 0;

  int ell = a.gamma;
  if (a.lengths) {
    ell = a.lengths[r];
    if (ell < 0 || ell > a.gamma) return;       // reported by the finish kernel
  }
  const bool pair = k < ell;
  const bool bonus = a.with_bonus && k == ell;
  if (!pair && !bonus) return;                   // same decision in every CTA of the cluster

  const Elem* trow = reinterpret_cast<const Elem*>(a.target) + (size_t(r) * a.Pt + k) * a.V;
  const Elem* drow = pair ? reinterpret_cast<const Elem*>(a.draft) + (size_t(r) * a.Pd + k) * a.V : nullptr;
  const int tile = int(rank) * NW + warp;
  const bool active = tile < a.nwt;

  S tq[VPT], tp[VPT];
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    if (active) tq[j].load(trow, slot_index<VPT, VW>(tile, j, lane), a.V);
    else tq[j].set_neg_inf();
  }
  auto load_draft = [&]() {
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      if (active && pair) tp[j].load(drow, slot_index<VPT, VW>(tile, j, lane), a.V);
      else tp[j].set_neg_inf();
    }
  };
  // with the draft exponentials kept in registers both rows are in flight at once;
  // otherwise the draft row is fetched after the target row's registers are free
  if constexpr (KEEP_P) load_draft();

  const float c2 = a.c2;
  // ---- pass 1, target row: tile max, exponentials (kept in shared memory), tile normaliser
  float mq = neg_inf();
#pragma unroll
  for (int j = 0; j < VPT; ++j) mq = fmaxf(mq, tq[j].vmax());
  mq = warp_max(mq);
  const bool q_live = mq > neg_inf();
  const float mq_c2 = q_live ? mq * c2 : 0.f;
  float zq = 0.f;
  float eq_reg[VEC ? 1 : NE];                    // unaligned path keeps them in registers
  if (q_live) {
    float2 za = make_float2(0.f, 0.f), zb = make_float2(0.f, 0.f);   // independent chains
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      if constexpr (VEC) {
#pragma unroll
        for (int h = 0; h < H; ++h) {
          const float2 t0 = fma2(make_float2(tq[j].get(4 * h), tq[j].get(4 * h + 1)), make_float2(c2, c2),
                                 make_float2(-mq_c2, -mq_c2));
          const float2 t1 = fma2(make_float2(tq[j].get(4 * h + 2), tq[j].get(4 * h + 3)), make_float2(c2, c2),
                                 make_float2(-mq_c2, -mq_c2));
          const float4 e = make_float4(ex2(t0.x), ex2(t0.y), ex2(t1.x), ex2(t1.y));
          za = add2(za, make_float2(e.x, e.y));
          zb = add2(zb, make_float2(e.z, e.w));
          s_exp[((warp * VPT + j) * H + h) * 32 + lane] = e;
        }
      } else {
        const float e = ex2(fmaf(tq[j].get(0), c2, -mq_c2));
        eq_reg[j] = e;
        if (j & 1) zb.x += e; else za.x += e;
      }
    }
    zq = warp_sum((za.x + za.y) + (zb.x + zb.y));
  }

  // ---- pass 1, draft row
  if constexpr (!KEEP_P) {
    asm volatile("" ::: "memory");
    load_draft();
  }
  float mp = neg_inf();
#pragma unroll
  for (int j = 0; j < VPT; ++j) mp = fmaxf(mp, tp[j].vmax());
  mp = warp_max(mp);
  const bool p_live = mp > neg_inf();
  const float mp_c2 = p_live ? mp * c2 : 0.f;
  // masked elements are -inf, so their exponentials are 0 without a select
  float ep[KEEP_P ? NE : 2];
  float zp = 0.f;
  {
    float2 za = make_float2(0.f, 0.f), zb = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < VPT; ++j)
#pragma unroll
      for (int e = 0; e < VW; e += (VW > 1 ? 2 : 1)) {
        if constexpr (VW > 1) {
          const float2 t = fma2(make_float2(tp[j].get(e), tp[j].get(e + 1)), make_float2(c2, c2),
                                make_float2(-mp_c2, -mp_c2));
          const float2 pe = make_float2(ex2(t.x), ex2(t.y));
          if constexpr (KEEP_P) {
            ep[j * VW + e] = pe.x;
            ep[j * VW + e + 1] = pe.y;
          }
          if ((e >> 1) & 1) zb = add2(zb, pe);
          else za = add2(za, pe);
        } else {
          const float pe = ex2(fmaf(tp[j].get(0), c2, -mp_c2));
          if constexpr (KEEP_P) ep[j] = pe;
          if (j & 1) zb.x += pe; else za.x += pe;
        }
      }
    if (p_live) zp = warp_sum((za.x + za.y) + (zb.x + zb.y));
  }

  // ---- CTA partial, then the row statistics across the cluster (distributed shared memory)
  if (lane == 0) s_warp[warp] = make_float4(q_live ? mq_c2 : neg_inf(), zq, p_live ? mp_c2 : neg_inf(), zp);
  __syncthreads();
  if (warp == 0) {
    const float4 w = lane < NW ? s_warp[lane] : make_float4(neg_inf(), 0.f, neg_inf(), 0.f);
    const float Mq = warp_max(w.x), Mp = warp_max(w.z);
    const float Zq = warp_sum(w.y > 0.f ? w.y * ex2(w.x - Mq) : 0.f);
    const float Zp = warp_sum(w.w > 0.f ? w.w * ex2(w.z - Mp) : 0.f);
    if (lane == 0) s_cta = make_float4(Mq, Zq, Mp, Zp);
    cluster_arrive_release();            // publishes s_cta to the cluster
  } else {
    cluster_arrive_relaxed();
  }
  cluster_wait_acquire();
  const float4 cp = lane < int(C) ? ld_shared_cluster_f4(cluster_map_shared(&s_cta, uint32_t(lane)))
                                  : make_float4(neg_inf(), 0.f, neg_inf(), 0.f);
  const float Mq = warp_max(cp.x), Mp = warp_max(cp.z);
  const float Zq = warp_sum(cp.y > 0.f ? cp.y * ex2(cp.x - Mq) : 0.f);
  const float Zp = warp_sum(cp.w > 0.f ? cp.w * ex2(cp.z - Mp) : 0.f);
  cluster_arrive_relaxed();              // this CTA's remote reads are done

  // ---- pass 2: tile residual mass sum [q - p]_+ = Q_tile - sum min(q, p), no second
  // exponential.  min(sq*eq, sp*ep) = s_hi * min(e_hi, rho * e_lo) with rho <= 1.
  const float sq = q_live ? tile_scale(mq_c2, Mq, Zq) : 0.f;
  const float sp = p_live ? tile_scale(mp_c2, Mp, Zp) : 0.f;
  float resid = 0.f;
  if (pair && q_live) {
    const bool q_hi = sq >= sp;
    const float rho = q_hi ? sp / sq : sq / sp;
    float2 aa = make_float2(0.f, 0.f), ab = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      if constexpr (VEC) {
#pragma unroll
        for (int h = 0; h < H; ++h) {
          const float4 e = s_exp[((warp * VPT + j) * H + h) * 32 + lane];
          float2 q0 = make_float2(e.x, e.y), q1 = make_float2(e.z, e.w);
          float2 p0, p1;
          if constexpr (KEEP_P) {
            const float* pe = ep + j * VW + 4 * h;
            p0 = make_float2(pe[0], pe[1]);
            p1 = make_float2(pe[2], pe[3]);
          } else {
            const float2 t0 = fma2(make_float2(tp[j].get(4 * h), tp[j].get(4 * h + 1)), make_float2(c2, c2),
                                   make_float2(-mp_c2, -mp_c2));
            const float2 t1 = fma2(make_float2(tp[j].get(4 * h + 2), tp[j].get(4 * h + 3)), make_float2(c2, c2),
                                   make_float2(-mp_c2, -mp_c2));
            p0 = make_float2(ex2(t0.x), ex2(t0.y));
            p1 = make_float2(ex2(t1.x), ex2(t1.y));
          }
          if (q_hi) {
            p0 = mul2(p0, make_float2(rho, rho));
            p1 = mul2(p1, make_float2(rho, rho));
          } else {
            q0 = mul2(q0, make_float2(rho, rho));
            q1 = mul2(q1, make_float2(rho, rho));
          }
          aa = add2(aa, make_float2(fminf(q0.x, p0.x), fminf(q0.y, p0.y)));
          ab = add2(ab, make_float2(fminf(q1.x, p1.x), fminf(q1.y, p1.y)));
        }
      } else {
        float epj;
        if constexpr (KEEP_P) epj = ep[j];
        else epj = ex2(fmaf(tp[j].get(0), c2, -mp_c2));
        const float qv = q_hi ? eq_reg[j] : eq_reg[j] * rho;
        const float pv = q_hi ? epj * rho : epj;
        if (j & 1) ab.x += fminf(qv, pv); else aa.x += fminf(qv, pv);
      }
    }
    const float mins = warp_sum((aa.x + aa.y) + (ab.x + ab.y)) * (q_hi ? sq : sp);
    resid = fmaxf(__fmul_rn(sq, zq) - mins, 0.f);
  }
  if (lane == 0 && active) {
    TileStats ts;
    ts.mq_c2 = q_live ? mq_c2 : neg_inf();
    ts.mp_c2 = p_live ? mp_c2 : neg_inf();
    ts.resid = resid;
    ts.qmass = __fmul_rn(sq, zq);
    a.tiles[size_t(item) * a.ntile_stride + tile] = ts;
  }
  if (rank == 0 && threadIdx.x == 0) {
    RowRec rr;
    rr.s.Mq_c2 = Mq; rr.s.Zq = Zq; rr.s.Mp_c2 = Mp; rr.s.Zp = Zp;
    a.rows[item] = rr;
  }
  cluster_wait_acquire();              // keep shared memory alive until every CTA has read it
}

// ---------------------------------------------------------------------------
// chain_stats, persistent and pipelined form for 16-byte-aligned rows.
//
// A grid of 8-CTA clusters sized to what fits at once (two 8-warp CTAs per
// SM); cluster c handles items c, c + n_clusters, ...  Every thread owns the
// same VPT slots of its warp tile in each row, and prefetches its slots of the
// next item into a private area of shared memory with 16-byte cp.async copies
// while the current item is processed from registers (no block-wide sync is
// needed for the staging: a thread only reads what it copied).  Pass 2
// recomputes the exponentials from the registers.  After pass 1 every warp
// stores its tile partial into each CTA of the cluster (distributed shared
// memory, double-buffered by the parity of the processed-item count), so one
// cluster barrier per item makes all partials local to every warp.
struct PipeArgs {
  StatsArgs s;
  int items;        // R * P
  int ncl;          // clusters in the grid
};

template <typename Elem, int VPT, int NW, bool COMPACT>
__global__ void __launch_bounds__(NW * 32, 2) chain_stats_pipe_kernel(PipeArgs pa) {
  using S = Slot<Elem, true>;
  constexpr int VW = S::VW;
  constexpr int kMaxParts = 8 * NW;             // cluster of at most 8 CTAs
  static_assert(kMaxParts <= 64, "two partials per lane");
  const StatsArgs& a = pa.s;
  extern __shared__ uint4 s_stage[];            // [2 rows][VPT][threads] (+ int[R + 1] when compacting)
  __shared__ float4 s_part[2][kMaxParts];       // every warp's partial of the cluster

  const uint32_t C = cluster_nctarank();
  const uint32_t rank = cluster_ctarank();
  const int cid = blockIdx.x / C;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = int(rank) * NW + warp;
  const bool active = tile < a.nwt;
  const long V = a.V;
  const float c2 = a.c2;
  if (cid == 0 && rank == 0 && threadIdx.x == 0) *reinterpret_cast<int*>(a.workspace) = 0;

  // this thread's slots: elements [base + j*32*VW, +VW) for j < jmax are in the row
  const long base = (long(tile) * 32 * VPT + lane) * VW;
  int jmax = 0;
  if (active && base < V) {
    const long n = (V - base + 32 * VW - 1) / (32 * VW);
    jmax = n < VPT ? int(n) : VPT;
  }

  // Items of this cluster: o = cid, cid + ncl, ...  Without compaction item o is
  // (o / P, o % P), decoded incrementally.  With ragged lengths (COMPACT) only
  // the live items are walked: the CTA scans n_r = l_r (+1 for the bonus row;
  // 0 for an invalid l_r) into s_pre and item o is (r, o - s_pre[r]) with
  // s_pre[r] <= o < s_pre[r+1].
  int n_items = pa.items;
  [[maybe_unused]] int* s_pre = reinterpret_cast<int*>(s_stage + 2 * VPT * NW * 32);
  if constexpr (COMPACT) {
    const int R = pa.items / a.P;
    const int per = (R + NW * 32 - 1) / (NW * 32);
    const int r0 = threadIdx.x * per, r1 = min(R, r0 + per);
    int cnt = 0;
    for (int q = r0; q < r1; ++q) {
      const int ell = __ldg(a.lengths + q);
      cnt += (ell >= 0 && ell <= a.gamma) ? ell + a.with_bonus : 0;
    }
    __shared__ int s_wsum[NW];
    const int lane_ = threadIdx.x & 31, warp_ = threadIdx.x >> 5;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane_ >= o) incl += t;
    }
    if (lane_ == 31) s_wsum[warp_] = incl;
    __syncthreads();
    int wpre = 0, total = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      if (w < warp_) wpre += s_wsum[w];
      total += s_wsum[w];
    }
    int run = wpre + incl - cnt;                 // live items before request r0
    for (int q = r0; q < r1; ++q) {
      s_pre[q] = run;
      const int ell = __ldg(a.lengths + q);
      run += (ell >= 0 && ell <= a.gamma) ? ell + a.with_bonus : 0;
    }
    if (threadIdx.x == 0) s_pre[R] = total;
    __syncthreads();
    n_items = total;
  }
  const int dr = pa.ncl / a.P, dk = pa.ncl - (pa.ncl / a.P) * a.P;
  auto advance = [&](int& r, int& k) {           // item + ncl, without compaction
    r += dr;
    k += dk;
    if (k >= a.P) { k -= a.P; ++r; }
  };
  auto locate = [&](int o, int& r, int& k) {     // item o, with compaction
    int lo = 0, hi = pa.items / a.P;             // s_pre[lo] <= o < s_pre[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_pre[mid] <= o) lo = mid;
      else hi = mid;
    }
    r = lo;
    k = o - s_pre[lo];
  };
  // Without compaction the walk visits (r, k') and processes position
  // k = (k' + r) mod P of request r.  Cluster c sees k' = (c + j * ncl) mod P;
  // when ncl shares a factor with P (36 clusters, P = 8) that is only a few
  // residues, so some clusters would get every cheap bonus row and others none.
  // Rotating each request's positions by r mixes them.
  auto rotate = [&](int r_, int k_) -> int {
    if constexpr (COMPACT) {
      return k_;
    } else {
      const int t = k_ + r_ % a.P;
      return t >= a.P ? t - a.P : t;
    }
  };
  auto kind_of = [&](int r, int k) -> int {      // 0 skip, 1 row pair, 2 bonus row
    int ell = a.gamma;
    if (a.lengths) {
      ell = __ldg(a.lengths + r);
      if (ell < 0 || ell > a.gamma) return 0;
    }
    if (k < ell) return 1;
    return (a.with_bonus && k == ell) ? 2 : 0;
  };
  auto stage = [&](int row, int j) -> uint4* { return s_stage + (row * VPT + j) * (NW * 32) + threadIdx.x; };
  auto copy_row = [&](int row, const Elem* src) {
    if (jmax == VPT) {
#pragma unroll
      for (int j = 0; j < VPT; ++j) cp_async16(stage(row, j), src + base + j * 32 * VW);
    } else {
#pragma unroll
      for (int j = 0; j < VPT; ++j)
        if (j < jmax) cp_async16(stage(row, j), src + base + j * 32 * VW);
    }
  };
  auto prefetch = [&](int item, int r, int kw) {
    if (item >= n_items || jmax == 0) return;
    const int k = rotate(r, kw);
    const int kind = kind_of(r, k);
    if (kind == 0) return;
    copy_row(0, reinterpret_cast<const Elem*>(a.target) + (size_t(r) * a.Pt + k) * size_t(V));
    if (kind == 1) copy_row(1, reinterpret_cast<const Elem*>(a.draft) + (size_t(r) * a.Pd + k) * size_t(V));
  };

  // Slots past the end of the row are never copied into: fill them with -inf
  // once, so that every item reads its slots without a per-slot select.
  {
    const uint32_t ninf = sizeof(Elem) == 2 ? (kBf16NegInf | (kBf16NegInf << 16)) : kF32NegInfBits;
#pragma unroll
    for (int j = 0; j < VPT; ++j)
      if (j >= jmax) {
        *stage(0, j) = make_uint4(ninf, ninf, ninf, ninf);
        *stage(1, j) = make_uint4(ninf, ninf, ninf, ninf);
      }
  }
  int r = 0, k = 0, rn = 0, kn = 0;                      // current and next item
  if constexpr (COMPACT) {
    if (cid < n_items) locate(cid, r, k);
    if (cid + pa.ncl < n_items) locate(cid + pa.ncl, rn, kn);
  } else {
    r = cid / a.P;
    k = cid - r * a.P;
    rn = r;
    kn = k;
    advance(rn, kn);
  }
  auto step_next = [&](int o, int& r2, int& k2) {  // (r2, k2) becomes item o + ncl
    if constexpr (COMPACT) {
      if (o + pa.ncl < n_items) locate(o + pa.ncl, r2, k2);
    } else {
      advance(r2, k2);
    }
  };
  prefetch(cid, r, k);
  cp_async_commit();
  int processed = 0;
  for (int o = cid; o < n_items; o += pa.ncl, r = rn, k = kn, step_next(o, rn, kn)) {
    const int kr = rotate(r, k);
    const int item = r * a.P + kr;                // storage index
    const int kind = kind_of(r, kr);
    cp_async_wait_all();                         // this thread's copies of `item` have landed
    // (the draft half of the stage is stale for a bonus row: its p results are dropped)
    S tq[VPT], tp[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const uint4 v = *stage(0, j);
      tq[j].w[0] = v.x; tq[j].w[1] = v.y; tq[j].w[2] = v.z; tq[j].w[3] = v.w;
      const uint4 u = *stage(1, j);
      tp[j].w[0] = u.x; tp[j].w[1] = u.y; tp[j].w[2] = u.z; tp[j].w[3] = u.w;
    }
    // tile maxima: consumes every staged value, so the slots are free to refill
    // (the refill is issued between the cluster barrier's arrive and wait)
    float mq = neg_inf(), mp = neg_inf();
    if constexpr (sizeof(Elem) == 2) {
      // pairwise (tree) reduction: a short dependency chain
      auto max2 = [](uint32_t x, uint32_t y) {
        uint32_t m;
        asm("max.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(x), "r"(y));
        return m;
      };
      auto slice_max = [&](const S* x) {
        uint32_t m[VPT];
#pragma unroll
        for (int j = 0; j < VPT; ++j) m[j] = max2(max2(x[j].w[0], x[j].w[1]), max2(x[j].w[2], x[j].w[3]));
#pragma unroll
        for (int st = 1; st < VPT; st <<= 1)
#pragma unroll
          for (int j = 0; j + st < VPT; j += 2 * st) m[j] = max2(m[j], m[j + st]);
        return fmaxf(__uint_as_float(m[0] << 16), __uint_as_float(m[0] & 0xFFFF0000u));
      };
      mq = slice_max(tq);
      mp = slice_max(tp);
    } else {
#pragma unroll
      for (int j = 0; j < VPT; ++j) {
        mq = fmaxf(mq, tq[j].vmax());
        mp = fmaxf(mp, tp[j].vmax());
      }
    }
    if (kind == 0) {
      prefetch(o + pa.ncl, rn, kn);
      cp_async_commit();
      continue;
    }
    if (kind == 2) mp = neg_inf();
    mq = warp_max(mq);
    mp = warp_max(mp);
    const bool q_live = mq > neg_inf();
    const bool p_live = mp > neg_inf();
    const float mq_c2 = q_live ? mq * c2 : 0.f;
    const float mp_c2 = p_live ? mp * c2 : 0.f;

    // ---- pass 1: tile normalisers for both rows (masked elements are -inf -> 0)
    auto tile_sum = [&](const S* x, float m_c2) -> float {
      float2 za = make_float2(0.f, 0.f), zb = za;
#pragma unroll
      for (int j = 0; j < VPT; ++j)
#pragma unroll
        for (int e = 0; e < VW; e += 4) {
          const float2 t0 = fma2(make_float2(x[j].get(e), x[j].get(e + 1)), make_float2(c2, c2), make_float2(-m_c2, -m_c2));
          za = add2(za, make_float2(ex2(t0.x), ex2(t0.y)));
          const float2 t1 = fma2(make_float2(x[j].get(e + 2), x[j].get(e + 3)), make_float2(c2, c2), make_float2(-m_c2, -m_c2));
          zb = add2(zb, make_float2(ex2(t1.x), ex2(t1.y)));
        }
      return (za.x + za.y) + (zb.x + zb.y);
    };
    float zq = 0.f, zp = 0.f;
    if (q_live) zq = tile_sum(tq, mq_c2);
    if (p_live) zp = tile_sum(tp, mp_c2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      zq += __shfl_xor_sync(0xffffffffu, zq, o);
      zp += __shfl_xor_sync(0xffffffffu, zp, o);
    }

    // ---- every warp's partial into every CTA, one cluster barrier, then the
    // row statistics from the C * NW local partials
    const int pb = processed & 1;
    {
      const float4 part = make_float4(q_live ? mq_c2 : neg_inf(), zq, p_live ? mp_c2 : neg_inf(), zp);
      if (lane < int(C)) st_shared_cluster_f4(cluster_map_shared(&s_part[pb][rank * NW + warp], uint32_t(lane)), part);
    }
    cluster_arrive_release();
    // The next item's copies are issued only now: issued before the arrive,
    // they held up its release fence.
    prefetch(o + pa.ncl, rn, kn);
    cp_async_commit();
    cluster_wait_acquire();
    const int nparts = int(C) * NW;
    const float4 none = make_float4(neg_inf(), 0.f, neg_inf(), 0.f);
    const float4 w0 = lane < nparts ? s_part[pb][lane] : none;
    const float4 w1 = lane + 32 < nparts ? s_part[pb][lane + 32] : none;
    const float Mq = warp_max(fmaxf(w0.x, w1.x)), Mp = warp_max(fmaxf(w0.z, w1.z));
    float Zq = (w0.y > 0.f ? w0.y * ex2(w0.x - Mq) : 0.f) + (w1.y > 0.f ? w1.y * ex2(w1.x - Mq) : 0.f);
    float Zp = (w0.w > 0.f ? w0.w * ex2(w0.z - Mp) : 0.f) + (w1.w > 0.f ? w1.w * ex2(w1.z - Mp) : 0.f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Zq += __shfl_xor_sync(0xffffffffu, Zq, o);
      Zp += __shfl_xor_sync(0xffffffffu, Zp, o);
    }

    // ---- pass 2: sum min(q, p) per tile with recomputed exponentials
    const float sq = q_live ? tile_scale(mq_c2, Mq, Zq) : 0.f;
    const float sp = p_live ? tile_scale(mp_c2, Mp, Zp) : 0.f;
    float resid = 0.f;
    if (kind == 1 && q_live) {
      // min(q, p) = 2^min(x_q*c2 + lq, x_p*c2 + lp): one exponential per position
      float lq, lp;
      asm("lg2.approx.f32 %0, %1;" : "=f"(lq) : "f"(sq));
      asm("lg2.approx.f32 %0, %1;" : "=f"(lp) : "f"(sp));
      lq -= mq_c2;
      lp = p_live ? lp - mp_c2 : neg_inf();
      float2 ma = make_float2(0.f, 0.f), mb = ma;
#pragma unroll
      for (int j = 0; j < VPT; ++j) {
        tq[j].launder();
        tp[j].launder();
      }
#pragma unroll
      for (int j = 0; j < VPT; ++j)
#pragma unroll
        for (int e = 0; e < VW; e += 2) {
          const float2 t = fma2(make_float2(tq[j].get(e), tq[j].get(e + 1)), make_float2(c2, c2),
                                make_float2(lq, lq));
          const float2 u = fma2(make_float2(tp[j].get(e), tp[j].get(e + 1)), make_float2(c2, c2),
                                make_float2(lp, lp));
          const float2 mn = make_float2(ex2(fminf(t.x, u.x)), ex2(fminf(t.y, u.y)));
          if ((e >> 1) & 1) mb = add2(mb, mn); else ma = add2(ma, mn);
        }
      float mins = (ma.x + ma.y) + (mb.x + mb.y);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mins += __shfl_xor_sync(0xffffffffu, mins, o);
      resid = fmaxf(__fmul_rn(sq, zq) - mins, 0.f);
    }
    if (lane == 0 && active) {
      TileStats ts;
      ts.mq_c2 = q_live ? mq_c2 : neg_inf();
      ts.mp_c2 = p_live ? mp_c2 : neg_inf();
      ts.resid = resid;
      ts.qmass = __fmul_rn(sq, zq);
      a.tiles[size_t(item) * a.ntile_stride + tile] = ts;
    }
    if (rank == 0 && threadIdx.x == 0) {
      RowRec rr;
      rr.s.Mq_c2 = Mq; rr.s.Zq = Zq; rr.s.Mp_c2 = Mp; rr.s.Zp = Zp;
      a.rows[item] = rr;
    }
    ++processed;
  }
  // No exit barrier is needed, because of one invariant: every CTA of a
  // cluster walks the same item sequence.  The walk depends only on the
  // cluster index, the grid's cluster count and the call's lengths (the
  // compacted walk's prefix is computed identically in every CTA from the same
  // lengths), and the kind of each item (skip, row pair, bonus row) is decided
  // from the same values, so every CTA executes the same number of cluster
  // barriers.  A CTA's last remote store into a peer's partials precedes its
  // arrive at the last barrier, and the peer reads them only after its wait,
  // so no CTA can exit while a peer may still store into its shared memory.
  // (Removing the per-item barrier breaks this: a remote store then can reach
  // a CTA that has already exited.)
  cp_async_wait_all();
  pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
struct FinishArgs {
  const void* target;
  const void* draft;
  const int32_t* tokens;      // [R, gamma]
  const int32_t* lengths;
  const float* uniforms;      // [R, gamma+1, 2]
  const RowRec* rows;
  const TileStats* tiles;
  void* workspace;
  int32_t* accepted;          // [R] or null (tv_accept)
  int32_t* out_token;
  float* c_star;              // [R, gamma] or null
  long V;
  int gamma, P, Pt, Pd;
  int nwt, ntile_stride;
  float c2;
  int sample;                 // 0: c* only (tv_accept)
};

// Per-element weight of the inverse-CDF draw: [q - p]_+ (rejection) or q
// (bonus), with the same arithmetic as chain_stats.
template <typename S>
__device__ __forceinline__ float draw_weight(const S& xq, const S& xp, int e, float c2, const TileStats& ts, float sq,
                                             float sp, bool q_live, bool p_live, bool use_resid) {
  if (!q_live) return 0.f;
  const float eq = ex2(fmaf(xq.get(e), c2, -ts.mq_c2));
  if (!use_resid) return __fmul_rn(eq, sq);
  const float ep = p_live ? ex2(fmaf(xp.get(e), c2, -ts.mp_c2)) : 0.f;
  return fmaxf(fmaf(eq, sq, -__fmul_rn(ep, sp)), 0.f);
}

// One CTA per request.  Phase 1, one warp per position k <= l_r in parallel:
// c*_k, the accept threshold min(1, q(x_k)/p(x_k)), and the tile a draw at k
// would come from (prefix over the tile masses: [q - p]_+ for k < l_r, q for
// the bonus position).  Phase 2: warp 0 finds the first rejection A by ballot.
// Phase 3: every warp rescans one slot of A's selected tile; a prefix over the
// slot totals picks the slot, one warp scan inside it picks the token.
template <typename Elem, bool VEC, int VPT>
__global__ void __launch_bounds__(kFinishThreads) chain_finish_kernel(FinishArgs a) {
  using S = Slot<Elem, VEC>;
  constexpr int VW = S::VW;
  constexpr int NWARP = kFinishThreads / 32;
  __shared__ float s_thr[SPECV_MAX_GAMMA + 1];
  __shared__ int s_sel[SPECV_MAX_GAMMA + 1];       // selected tile (-1: none)
  __shared__ float s_base[SPECV_MAX_GAMMA + 1];    // mass before that tile
  __shared__ float s_target[SPECV_MAX_GAMMA + 1];  // u * total mass
  __shared__ int s_resid[SPECV_MAX_GAMMA + 1];     // draw from [q-p]_+ (1) or q (0)
  __shared__ float s_slot[VPT];
  __shared__ int s_slot_last[VPT];
  __shared__ int s_bad, s_A, s_tok;
  pdl_wait_primary();
  const int r = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gamma = a.gamma;
  int ell = a.lengths ? __ldg(a.lengths + r) : gamma;
  const bool bad_len = ell < 0 || ell > gamma;
  if (bad_len) ell = 0;
  if (threadIdx.x == 0) {
    s_bad = bad_len ? 1 : 0;
    s_tok = -1;
  }
  __syncthreads();

  // ---- phase 1
  const int kmax = a.sample ? ell : ell - 1;
  for (int k = warp; k <= kmax && !bad_len; k += NWARP) {
    const int item = r * a.P + k;
    const TileStats* ts = a.tiles + size_t(item) * a.ntile_stride;
    const bool pair = k < ell;
    const int per = (a.nwt + 31) / 32;            // consecutive tiles per lane (index order), <= 4
    const int t0 = lane * per, t1 = min(a.nwt, t0 + per);
    float tres[kMaxTiles / 32], tqm[kMaxTiles / 32];
    float rsum = 0.f, qsum = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxTiles / 32; ++i) {
      tres[i] = 0.f;
      tqm[i] = 0.f;
      if (t0 + i < t1) {
        const TileStats x = ts[t0 + i];
        tres[i] = x.resid;
        tqm[i] = x.qmass;
      }
      rsum += tres[i];
      qsum += tqm[i];
    }
    int x = 0;
    float u0 = 0.f, u1 = 0.f;
    if (a.sample) {
      if (pair) x = __ldg(a.tokens + size_t(r) * gamma + k);
      u0 = __ldg(a.uniforms + (size_t(r) * (gamma + 1) + k) * 2);
      u1 = __ldg(a.uniforms + (size_t(r) * (gamma + 1) + k) * 2 + 1);
    }
    const float resid_total = warp_sum(rsum);
    if (pair && a.c_star && lane == 0) a.c_star[size_t(r) * gamma + k] = 1.f - resid_total;
    if (!a.sample) continue;
    const bool bad = !(u1 >= 0.f && u1 < 1.f) || (pair && !(u0 >= 0.f && u0 < 1.f)) || (pair && !(x >= 0 && x < a.V));
    // the tile a draw at k comes from
    bool use_resid = pair;
    float lsum = use_resid ? rsum : qsum;
    float incl = warp_inclusive_scan(lsum);
    float total = __shfl_sync(0xffffffffu, incl, 31);
    if (use_resid && !(total > 0.f)) {            // no residual mass: draw from q
      use_resid = false;
      lsum = qsum;
      incl = warp_inclusive_scan(lsum);
      total = __shfl_sync(0xffffffffu, incl, 31);
    }
    const float target = u1 * total;
    const unsigned hit = __ballot_sync(0xffffffffu, incl > target && t1 > t0);
    int sel_tile = -1;
    float base = 0.f;
    {
      const int L = hit ? __ffs(hit) - 1 : 31;
      if (lane == L) {
        // first tile of this lane whose running sum passes the target; if rounding
        // leaves none, the lane's last tile with mass
        float run = incl - lsum;
        bool found = false;
#pragma unroll
        for (int i = 0; i < kMaxTiles / 32; ++i) {
          const float m = use_resid ? tres[i] : tqm[i];
          if (!found && t0 + i < t1 && m > 0.f) {
            sel_tile = t0 + i;
            base = run;
            found = hit && run + m > target;
          }
          if (!found) run += m;
        }
      }
      sel_tile = __shfl_sync(0xffffffffu, sel_tile, L);
      base = __shfl_sync(0xffffffffu, base, L);
    }
    // accept threshold from the draft token's two logits
    float thr = 1.f;
    if (pair && !bad && lane == 0) {
      const RowStats rs = a.rows[item].s;
      const size_t iq = (size_t(r) * a.Pt + k) * size_t(a.V) + x;
      const size_t ip = (size_t(r) * a.Pd + k) * size_t(a.V) + x;
      float lq, lp;
      if constexpr (sizeof(Elem) == 2) {
        lq = __uint_as_float(uint32_t(__ldg(reinterpret_cast<const unsigned short*>(a.target) + iq)) << 16);
        lp = __uint_as_float(uint32_t(__ldg(reinterpret_cast<const unsigned short*>(a.draft) + ip)) << 16);
      } else {
        lq = __ldg(reinterpret_cast<const float*>(a.target) + iq);
        lp = __ldg(reinterpret_cast<const float*>(a.draft) + ip);
      }
      const float qx = ex2(fmaf(lq, a.c2, -rs.Mq_c2)) / rs.Zq;
      const float px = ex2(fmaf(lp, a.c2, -rs.Mp_c2)) / rs.Zp;
      thr = px > 0.f ? fminf(1.f, qx / px) : 1.f;
    }
    if (lane == 0) {
      s_thr[k] = thr;
      s_sel[k] = sel_tile;
      s_base[k] = base;
      s_target[k] = target;
      s_resid[k] = use_resid ? 1 : 0;
      if (bad) s_bad = 1;
    }
  }
  if (a.c_star && lane == 0)
    for (int k = warp; k < gamma; k += NWARP)
      if (bad_len || k >= ell) a.c_star[size_t(r) * gamma + k] = __int_as_float(0x7fc00000);
  if (!a.sample) return;
  __syncthreads();

  // ---- phase 2: first rejection
  if (warp == 0) {
    bool rej = false;
    if (!bad_len && lane < ell) {
      const float u0 = __ldg(a.uniforms + (size_t(r) * (gamma + 1) + lane) * 2);
      rej = !(u0 < s_thr[lane]);
    }
    const unsigned rm = __ballot_sync(0xffffffffu, rej);
    if (lane == 0) s_A = rm ? __ffs(rm) - 1 : ell;
  }
  __syncthreads();
  const int A = s_A;
  const int tile = s_bad ? -1 : s_sel[A];

  // ---- phase 3: rescan A's selected tile, one slot per warp
  if (tile >= 0) {
    const int item = r * a.P + A;
    const bool use_resid = s_resid[A] != 0;
    const TileStats tsr = a.tiles[size_t(item) * a.ntile_stride + tile];
    const RowStats rs = a.rows[item].s;
    const Elem* trow = reinterpret_cast<const Elem*>(a.target) + (size_t(r) * a.Pt + A) * a.V;
    const Elem* drow = use_resid ? reinterpret_cast<const Elem*>(a.draft) + (size_t(r) * a.Pd + A) * a.V : nullptr;
    const bool q_live = tsr.mq_c2 > neg_inf();
    const bool p_live = use_resid && tsr.mp_c2 > neg_inf();
    const float sq = q_live ? tile_scale(tsr.mq_c2, rs.Mq_c2, rs.Zq) : 0.f;
    const float sp = p_live ? tile_scale(tsr.mp_c2, rs.Mp_c2, rs.Zp) : 0.f;
    float w[(VPT + NWARP - 1) / NWARP][VW];
#pragma unroll
    for (int i = 0; i < (VPT + NWARP - 1) / NWARP; ++i) {
      const int j = warp + i * NWARP;
      if (j < VPT) {
        S xq, xp;
        const long idx0 = slot_index<VPT, VW>(tile, j, lane);
        xq.load(trow, idx0, a.V);
        if (use_resid) xp.load(drow, idx0, a.V);
        else xp.set_neg_inf();
        float sum = 0.f;
        int last = -1;
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          w[i][e] = draw_weight(xq, xp, e, a.c2, tsr, sq, sp, q_live, p_live, use_resid);
          sum += w[i][e];
          if (w[i][e] > 0.f) last = int(idx0) + e;
        }
        const float total = warp_sum(sum);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
        if (lane == 0) {
          s_slot[j] = total;
          s_slot_last[j] = last;
        }
      }
    }
    __syncthreads();
    // slot holding the target (every warp computes the same answer)
    const float target = s_target[A];
    float run = s_base[A];
    int js = -1, jlast = -1, last_any = -1;
    for (int j = 0; j < VPT; ++j) {
      if (s_slot_last[j] >= 0) { jlast = j; last_any = s_slot_last[j]; }
      if (js < 0 && run + s_slot[j] > target && s_slot[j] > 0.f) js = j;
      else if (js < 0) run += s_slot[j];
    }
    if (js < 0) {                                  // rounding at the top: the tile's last positive weight
      if (threadIdx.x == 0) s_tok = last_any;
    } else if (warp == js % NWARP) {
      const int i = js / NWARP;
      float lsum = 0.f;
#pragma unroll
      for (int ii = 0; ii < (VPT + NWARP - 1) / NWARP; ++ii)
        if (ii == i)
#pragma unroll
          for (int e = 0; e < VW; ++e) lsum += w[ii][e];
      const float incl = warp_inclusive_scan(lsum);
      float acc = run + (incl - lsum);
      int cand = 0x7fffffff;
      const long idx0 = slot_index<VPT, VW>(tile, js, lane);
#pragma unroll
      for (int ii = 0; ii < (VPT + NWARP - 1) / NWARP; ++ii)
        if (ii == i)
#pragma unroll
          for (int e = 0; e < VW; ++e) {
            acc += w[ii][e];
            if (cand == 0x7fffffff && acc > target && w[ii][e] > 0.f) cand = int(idx0) + e;
          }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
      if (lane == 0) s_tok = cand != 0x7fffffff ? cand : s_slot_last[js];
    }
    (void)jlast;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int tok = s_tok;
    const bool bad = s_bad != 0 || tok < 0;
    a.accepted[r] = bad ? -1 : A;
    a.out_token[r] = bad ? -1 : tok;
    if (bad) record_device_error(a.workspace, SPECV_ERR_DEVICE_DATA);
  }
}

// ---------------------------------------------------------------------------
// argmax per warp tile
struct ArgmaxArgs {
  const void* logits;
  const int32_t* lengths;     // rows k > lengths[r] + lim_off are skipped (null: none skipped)
  void* workspace;
  ArgRec* out;                // [R * Pout, ntile_stride]
  long V;
  int P;                      // rows per request in the logits tensor
  int Pout;                   // rows per request processed (k < Pout) = output stride
  int lim_off;
  int gamma;                  // bound for lengths
  int nwt, ntile_stride;
  int clear_error;
};

template <typename Elem, bool VEC, int VPT>
__global__ void __launch_bounds__(kArgmaxWarps * 32) argmax_tiles_kernel(ArgmaxArgs a) {
  using S = Slot<Elem, VEC>;
  constexpr int VW = S::VW;
  const int item = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.y * kArgmaxWarps + warp;
  if (a.clear_error && item == 0 && blockIdx.y == 0 && threadIdx.x == 0) *reinterpret_cast<int*>(a.workspace) = 0;
  if (tile >= a.nwt) return;
  const int r = item / a.Pout, k = item - r * a.Pout;
  if (a.lengths) {
    const int ell = a.lengths[r];
    if (ell < 0 || ell > a.gamma || k > ell + a.lim_off) return;
  }
  const Elem* row = reinterpret_cast<const Elem*>(a.logits) + (size_t(r) * a.P + k) * a.V;
  S x[VPT];
#pragma unroll
  for (int j = 0; j < VPT; ++j) x[j].load(row, slot_index<VPT, VW>(tile, j, lane), a.V);
  float m = neg_inf();
#pragma unroll
  for (int j = 0; j < VPT; ++j) m = fmaxf(m, x[j].vmax());
  int idx = 0x7fffffff;
#pragma unroll
  for (int j = VPT - 1; j >= 0; --j)
#pragma unroll
    for (int e = VW - 1; e >= 0; --e)
      if (x[j].get(e) == m) idx = int(slot_index<VPT, VW>(tile, j, lane)) + e;
  warp_argmax(m, idx);
  if (lane == 0) {
    ArgRec ar;
    ar.v = m;
    ar.i = idx;
    a.out[size_t(item) * a.ntile_stride + tile] = ar;
  }
  pdl_launch_dependents();
}

struct GreedyArgs {
  const int32_t* tokens;
  const int32_t* lengths;
  const ArgRec* targ;         // [R*tpos, stride]
  const ArgRec* darg;         // [R*gamma, stride] or null
  void* workspace;
  int32_t* accepted;
  int32_t* out_token;
  float* c_star;
  long V;
  int gamma, tpos, nwt, ntile_stride;
  int sample;
};

// One CTA per request, one warp per position: g_k = argmax target row k (and
// the draft argmax for c*), then warp 0 finds the first mismatch by ballot.
constexpr int kGreedyThreads = 256;

__global__ void __launch_bounds__(kGreedyThreads) greedy_finish_kernel(GreedyArgs a) {
  constexpr int NW = kGreedyThreads / 32;
  __shared__ int s_g[SPECV_MAX_GAMMA + 1], s_gd[SPECV_MAX_GAMMA];
  pdl_wait_primary();                      // the argmax tile records are complete
  const int r = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gamma = a.gamma;
  int ell = a.lengths ? __ldg(a.lengths + r) : gamma;
  const bool bad_len = ell < 0 || ell > gamma;
  if (bad_len) ell = 0;
  const int kt = a.sample ? ell : ell - 1;             // target rows used: 0 .. kt
  for (int k = warp; k <= gamma; k += NW) {
    int g = -1, gd = -1;
    if (!bad_len && k <= kt) g = combine_argmax(a.targ + size_t(r * a.tpos + k) * a.ntile_stride, a.nwt);
    if (!bad_len && a.darg && k < ell) gd = combine_argmax(a.darg + size_t(r * gamma + k) * a.ntile_stride, a.nwt);
    if (lane == 0) {
      s_g[k] = g;
      if (k < gamma) s_gd[k] = gd;
    }
  }
  __syncthreads();
  if (a.c_star)
    for (int k = threadIdx.x; k < gamma; k += kGreedyThreads)
      a.c_star[size_t(r) * gamma + k] =
          (!bad_len && k < ell) ? ((s_gd[k] == s_g[k]) ? 1.f : 0.f) : __int_as_float(0x7fc00000);
  if (!a.sample || warp != 0) return;
  bool mismatch = false, valid = true;
  if (lane < ell) {
    const int x = __ldg(a.tokens + size_t(r) * gamma + lane);
    valid = x >= 0 && x < a.V;
    mismatch = x != s_g[lane];
  }
  const bool bad = bad_len || __any_sync(0xffffffffu, !valid);
  const unsigned mm = __ballot_sync(0xffffffffu, mismatch);
  const int A = mm ? __ffs(mm) - 1 : ell;
  // correction (A < l_r) or bonus (A = l_r) token: the target argmax of row A
  if (lane == 0) {
    a.accepted[r] = bad ? -1 : A;
    a.out_token[r] = bad ? -1 : s_g[A];
    if (bad) record_device_error(a.workspace, SPECV_ERR_DEVICE_DATA);
  }
}

// ---------------------------------------------------------------------------
// host side

namespace {

// One tiling choice for a row length V.
struct Tiling {
  int vec;          // 1: 16-byte vectors
  int vpt;          // vectors (slots) per lane per row
  int vw;           // elements per slot
  int nwt;          // warp tiles per row
  int cluster;      // CTAs per row (chain_stats)
  int stride;       // tile records per row in the workspace
  int warps;        // warps (tiles) per CTA in chain_stats
  int pipe;         // 1: persistent pipelined chain_stats
};

constexpr int kVptList[] = {1, 2, 4, 6, 8, 10};

// 8-warp CTAs: the unaligned path and the argmax / greedy path
bool choose_tiling(long V, specv_dtype dtype, bool vec_ok, Tiling* t) {
  const int vw = vec_ok ? (dtype == SPECV_BF16 ? 8 : 4) : 1;
  for (int pass = 0; pass < 2; ++pass) {
    const int cmax = pass == 0 ? 8 : kMaxCluster;
    for (int vpt : kVptList) {
      const long tile = 32L * vpt * vw;
      const long nwt = (V + tile - 1) / tile;
      const long cl = (nwt + kStatsWarps - 1) / kStatsWarps;
      if (cl <= cmax) {
        t->vec = vec_ok ? 1 : 0;
        t->vpt = vpt;
        t->vw = vw;
        t->nwt = int(nwt);
        t->cluster = int(cl);
        t->stride = int(cl) * kStatsWarps;
        t->warps = kStatsWarps;
        t->pipe = 0;
        return true;
      }
    }
  }
  return false;
}

// Persistent pipelined kernel: 16-byte rows, up to 8 CTAs per cluster of
// kPipeWarps warps each, two CTAs per SM (measured fastest of the persistent
// and non-persistent forms tried for the 151936-token workload).
constexpr int kPipeWarps = 8;
constexpr int kPipeVptBf16[] = {1, 2, 4, 6, 8, 10};
constexpr int kPipeVptF32[] = {2, 4, 6, 8, 10};

bool choose_pipe(long V, specv_dtype dtype, bool vec_ok, Tiling* t) {
  if (!vec_ok) return false;
  const int vw = dtype == SPECV_BF16 ? 8 : 4;
  const int* list = dtype == SPECV_BF16 ? kPipeVptBf16 : kPipeVptF32;
  const int nlist = dtype == SPECV_BF16 ? int(sizeof(kPipeVptBf16) / sizeof(int)) : int(sizeof(kPipeVptF32) / sizeof(int));
  for (int i = 0; i < nlist; ++i) {
    const long tile = 32L * list[i] * vw;
    const long nwt = (V + tile - 1) / tile;
    const long cl = (nwt + kPipeWarps - 1) / kPipeWarps;
    if (cl <= 8) {
      t->vec = 1;
      t->vpt = list[i];
      t->vw = vw;
      t->nwt = int(nwt);
      t->cluster = int(cl);
      t->stride = int(cl) * kPipeWarps;
      t->warps = kPipeWarps;
      t->pipe = 1;
      return true;
    }
  }
  return false;
}

// the tiling a T > 0 call uses
bool choose_sampling_tiling(long V, specv_dtype dtype, bool vec_ok, Tiling* t) {
  return choose_pipe(V, dtype, vec_ok, t) || choose_tiling(V, dtype, vec_ok, t);
}

template <typename Elem, bool VEC, int VPT>
struct ChainKernels {
  static void* stats() { return reinterpret_cast<void*>(&chain_stats_kernel<Elem, VEC, VPT, kStatsWarps, true>); }
  static void* finish() { return reinterpret_cast<void*>(&chain_finish_kernel<Elem, VEC, VPT>); }
  static void* argmax() { return reinterpret_cast<void*>(&argmax_tiles_kernel<Elem, VEC, VPT>); }
};

struct KernelSet {
  void* stats;
  void* finish;
  void* argmax;
  void* stats_compact;        // persistent form walking only the live items of ragged lengths
};

template <typename Elem, bool VEC>
KernelSet pick_vpt(int vpt) {
  switch (vpt) {
    case 1: return {ChainKernels<Elem, VEC, 1>::stats(), ChainKernels<Elem, VEC, 1>::finish(), ChainKernels<Elem, VEC, 1>::argmax()};
    case 2: return {ChainKernels<Elem, VEC, 2>::stats(), ChainKernels<Elem, VEC, 2>::finish(), ChainKernels<Elem, VEC, 2>::argmax()};
    case 4: return {ChainKernels<Elem, VEC, 4>::stats(), ChainKernels<Elem, VEC, 4>::finish(), ChainKernels<Elem, VEC, 4>::argmax()};
    case 6: return {ChainKernels<Elem, VEC, 6>::stats(), ChainKernels<Elem, VEC, 6>::finish(), ChainKernels<Elem, VEC, 6>::argmax()};
    case 8: return {ChainKernels<Elem, VEC, 8>::stats(), ChainKernels<Elem, VEC, 8>::finish(), ChainKernels<Elem, VEC, 8>::argmax()};
    default: return {ChainKernels<Elem, VEC, 10>::stats(), ChainKernels<Elem, VEC, 10>::finish(), ChainKernels<Elem, VEC, 10>::argmax()};
  }
}

template <typename Elem, int VPT>
KernelSet pipe_set() {
  return {reinterpret_cast<void*>(&chain_stats_pipe_kernel<Elem, VPT, kPipeWarps, false>),
          reinterpret_cast<void*>(&chain_finish_kernel<Elem, true, VPT>), nullptr,
          reinterpret_cast<void*>(&chain_stats_pipe_kernel<Elem, VPT, kPipeWarps, true>)};
}

// clusters of the persistent kernel that fit at once, cached per device and kernel
int max_active_clusters(void* fn, size_t smem, int cluster, int threads) {
  constexpr int kSlots = 32;
  static std::atomic<uintptr_t> keys[kSlots];
  static std::atomic<int> vals[kSlots];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const uintptr_t key = (reinterpret_cast<uintptr_t>(fn) ^ (uintptr_t(dev) << 48) ^ (uintptr_t(cluster) << 56)) | 1;
  for (int i = 0; i < kSlots; ++i)
    if (keys[i].load(std::memory_order_acquire) == key) return vals[i].load(std::memory_order_relaxed);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(cluster) * 64);
  cfg.blockDim = dim3(unsigned(threads));
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = unsigned(cluster);
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) n = 0;
  for (int i = 0; i < kSlots; ++i) {
    uintptr_t expected = 0;
    if (keys[i].load(std::memory_order_relaxed) == 0 && keys[i].compare_exchange_strong(expected, key)) {
      vals[i].store(n, std::memory_order_relaxed);
      break;
    }
  }
  return n;
}

KernelSet kernels_for(specv_dtype dtype, const Tiling& t) {
  if (t.pipe) {
    if (dtype == SPECV_BF16)
      switch (t.vpt) {
        case 1: return pipe_set<uint16_t, 1>();
        case 2: return pipe_set<uint16_t, 2>();
        case 4: return pipe_set<uint16_t, 4>();
        case 6: return pipe_set<uint16_t, 6>();
        case 8: return pipe_set<uint16_t, 8>();
        default: return pipe_set<uint16_t, 10>();
      }
    switch (t.vpt) {
      case 2: return pipe_set<float, 2>();
      case 4: return pipe_set<float, 4>();
      case 6: return pipe_set<float, 6>();
      case 8: return pipe_set<float, 8>();
      default: return pipe_set<float, 10>();
    }
  }
  if (dtype == SPECV_BF16) return t.vec ? pick_vpt<uint16_t, true>(t.vpt) : pick_vpt<uint16_t, false>(t.vpt);
  return t.vec ? pick_vpt<float, true>(t.vpt) : pick_vpt<float, false>(t.vpt);
}

// Workspace: header | rows RowRec[items] | then either (T > 0) tiles
// TileStats[items][ntile_stride], or (T = 0) target argmax
// ArgRec[R*(gamma+1)][stride] | draft argmax ArgRec[R*gamma][stride].  A call
// takes one of the two paths, so the two regions share their bytes.
struct ChainLayout {
  size_t rows_off, tiles_off, targ_off, darg_off, total;
  int ntile_stride;
};

ChainLayout chain_layout(int R, int gamma, const Tiling& t) {
  ChainLayout L;
  L.ntile_stride = t.stride;
  const size_t items = size_t(R) * (gamma + 1);
  size_t off = kHeaderBytes;
  L.rows_off = off;
  off = align256(off + items * sizeof(RowRec));
  L.tiles_off = off;
  L.targ_off = off;
  const size_t tiles_end = align256(off + items * L.ntile_stride * sizeof(TileStats));
  L.darg_off = align256(off + items * L.ntile_stride * sizeof(ArgRec));
  const size_t darg_end = align256(L.darg_off + size_t(R) * gamma * L.ntile_stride * sizeof(ArgRec));
  L.total = tiles_end > darg_end ? tiles_end : darg_end;
  return L;
}

bool rows_vector_ok(const void* p, long V, specv_dtype dtype) {
  const int vw = dtype == SPECV_BF16 ? 8 : 4;
  return p == nullptr || ((reinterpret_cast<uintptr_t>(p) & 15) == 0 && V % vw == 0);
}

specv_status launch_stats(const KernelSet& ks, const Tiling& t, const StatsArgs& sa, int items, cudaStream_t st,
                          specv_dtype dtype) {
  if (items == 0) return SPECV_OK;
  if (t.pipe) {
    const int R = items / sa.P;
    const bool compact = sa.lengths != nullptr && R <= kMaxCompactRequests;
    void* fn = compact ? ks.stats_compact : ks.stats;
    const size_t smem = size_t(2) * t.vpt * t.warps * 32 * sizeof(uint4) + (compact ? size_t(R + 1) * sizeof(int) : 0);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
      return SPECV_ERR_CUDA;
    const int maxcl = max_active_clusters(fn, smem, t.cluster, t.warps * 32);
    if (maxcl < 1) return SPECV_ERR_UNSUPPORTED;
    PipeArgs pa;
    pa.s = sa;
    pa.items = items;
    pa.ncl = items < maxcl ? items : maxcl;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(pa.ncl) * unsigned(t.cluster));
    cfg.blockDim = dim3(unsigned(t.warps) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = unsigned(t.cluster);
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    void* args[] = {&pa};
    if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) return SPECV_ERR_CUDA;
    return SPECV_OK;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(items) * unsigned(t.cluster));
  cfg.blockDim = dim3(unsigned(t.warps) * 32);
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = unsigned(t.cluster);
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (t.cluster > 8) {
    if (cudaFuncSetAttribute(ks.stats, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      return SPECV_ERR_CUDA;
  }
  const size_t smem = t.vec ? size_t(t.warps) * t.vpt * (t.vw / 4) * 32 * sizeof(float4) : 0;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(ks.stats, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
    return SPECV_ERR_CUDA;
  cfg.dynamicSmemBytes = smem;
  void* args[] = {const_cast<StatsArgs*>(&sa)};
  if (cudaLaunchKernelExC(&cfg, ks.stats, args) != cudaSuccess) return SPECV_ERR_CUDA;
  return SPECV_OK;
}

}  // namespace

// T > 0 shared front half: chain_stats over `items` row pairs
static specv_status chain_sampling(const void* target, const void* draft, specv_dtype dtype, const int32_t* tokens,
                                   const int32_t* lengths, const float* uniforms, int R, int gamma, int P, int Pt,
                                   int Pd, long V, float T, int32_t* accepted, int32_t* out_token, float* c_star,
                                   void* ws, const Tiling& t, cudaStream_t st, bool sample) {
  const ChainLayout L = chain_layout(R, gamma, t);
  const KernelSet ks = kernels_for(dtype, t);
  char* base = static_cast<char*>(ws);
  StatsArgs sa;
  sa.target = target;
  sa.draft = draft;
  sa.tokens = tokens;
  sa.lengths = lengths;
  sa.workspace = ws;
  sa.rows = reinterpret_cast<RowRec*>(base + L.rows_off);
  sa.tiles = reinterpret_cast<TileStats*>(base + L.tiles_off);
  sa.V = V;
  sa.gamma = gamma;
  sa.P = P;
  sa.Pt = Pt;
  sa.Pd = Pd;
  sa.nwt = t.nwt;
  sa.ntile_stride = L.ntile_stride;
  sa.with_bonus = sample ? 1 : 0;
  sa.c2 = kLog2e / T;
  specv_status s = launch_stats(ks, t, sa, R * P, st, dtype);
  if (s != SPECV_OK) return s;
  FinishArgs fa;
  fa.target = target;
  fa.draft = draft;
  fa.tokens = tokens;
  fa.lengths = lengths;
  fa.uniforms = uniforms;
  fa.rows = sa.rows;
  fa.tiles = sa.tiles;
  fa.workspace = ws;
  fa.accepted = accepted;
  fa.out_token = out_token;
  fa.c_star = c_star;
  fa.V = V;
  fa.gamma = gamma;
  fa.P = P;
  fa.Pt = Pt;
  fa.Pd = Pd;
  fa.nwt = t.nwt;
  fa.ntile_stride = L.ntile_stride;
  fa.c2 = sa.c2;
  fa.sample = sample ? 1 : 0;
  void* fargs[] = {&fa};
  // programmatic dependent launch: the finish grid is scheduled while the stats
  // grid drains and waits (griddepcontrol.wait) for its results
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(R));
  cfg.blockDim = dim3(kFinishThreads);
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelExC(&cfg, ks.finish, fargs) != cudaSuccess) return SPECV_ERR_CUDA;
  return SPECV_OK;
}

static specv_status launch_argmax(const KernelSet& ks, const Tiling& t, const void* logits, const int32_t* lengths,
                                  void* ws, ArgRec* out, int R, int P, int Pout, int lim_off, int gamma, long V,
                                  int ntile_stride, bool clear_error, cudaStream_t st) {
  ArgmaxArgs aa;
  aa.logits = logits;
  aa.lengths = lengths;
  aa.workspace = ws;
  aa.out = out;
  aa.V = V;
  aa.P = P;
  aa.Pout = Pout;
  aa.lim_off = lim_off;
  aa.gamma = gamma;
  aa.nwt = t.nwt;
  aa.ntile_stride = ntile_stride;
  aa.clear_error = clear_error ? 1 : 0;
  void* args[] = {&aa};
  const unsigned ctas_per_row = unsigned((t.nwt + kArgmaxWarps - 1) / kArgmaxWarps);
  if (cudaLaunchKernel(ks.argmax, dim3(unsigned(R) * unsigned(Pout), ctas_per_row), dim3(kArgmaxWarps * 32), args, 0,
                       st) != cudaSuccess)
    return SPECV_ERR_CUDA;
  return SPECV_OK;
}

// T = 0.  sample: verify_chain (target rows k <= l_r, draft rows k < l_r when c* is
// wanted); otherwise tv_accept (rows k < gamma of a target tensor with Pt rows per request).
static specv_status chain_greedy(const void* target, const void* draft, specv_dtype dtype, const int32_t* tokens,
                                 const int32_t* lengths, int R, int gamma, int Pt, long V, int32_t* accepted,
                                 int32_t* out_token, float* c_star, void* ws, const Tiling& t, cudaStream_t st,
                                 bool sample) {
  const ChainLayout L = chain_layout(R, gamma, t);
  const KernelSet ks = kernels_for(dtype, t);
  char* base = static_cast<char*>(ws);
  ArgRec* targ = reinterpret_cast<ArgRec*>(base + L.targ_off);
  ArgRec* darg = reinterpret_cast<ArgRec*>(base + L.darg_off);
  const int tpos = sample ? gamma + 1 : gamma;
  specv_status s = launch_argmax(ks, t, target, sample ? lengths : nullptr, ws, targ, R, Pt, tpos, 0, gamma, V,
                                 L.ntile_stride, true, st);
  if (s != SPECV_OK) return s;
  if (c_star && gamma > 0) {
    s = launch_argmax(ks, t, draft, sample ? lengths : nullptr, ws, darg, R, gamma, gamma, -1, gamma, V,
                      L.ntile_stride, false, st);
    if (s != SPECV_OK) return s;
  }
  GreedyArgs ga;
  ga.tokens = tokens;
  ga.lengths = sample ? lengths : nullptr;
  ga.targ = targ;
  ga.darg = c_star ? darg : nullptr;
  ga.workspace = ws;
  ga.accepted = accepted;
  ga.out_token = out_token;
  ga.c_star = c_star;
  ga.V = V;
  ga.gamma = gamma;
  ga.tpos = tpos;
  ga.nwt = t.nwt;
  ga.ntile_stride = L.ntile_stride;
  ga.sample = sample ? 1 : 0;
  void* gargs[] = {&ga};
  if (launch_dependent(reinterpret_cast<void*>(&greedy_finish_kernel), dim3(R), dim3(kGreedyThreads), gargs, st) !=
      cudaSuccess)
    return SPECV_ERR_CUDA;
  return SPECV_OK;
}


// ---------------------------------------------------------------------------
// argmax over rows, exported for the tree verifier
bool argmax_plan(long V, specv_dtype dtype, bool vec_ok, ArgmaxPlan* p) {
  Tiling t;
  if (!choose_tiling(V, dtype, vec_ok, &t)) return false;
  p->vec = t.vec;
  p->vpt = t.vpt;
  p->nwt = t.nwt;
  p->stride = t.cluster * kStatsWarps;
  return true;
}

specv_status launch_argmax_rows(const ArgmaxPlan& p, specv_dtype dtype, const void* logits, int R, int P, int Pout,
                                const int32_t* lengths, int lim_off, int gamma, long V, void* ws, ArgRec* out,
                                bool clear_error, cudaStream_t st) {
  Tiling t;
  t.vec = p.vec;
  t.vpt = p.vpt;
  t.vw = 0;
  t.nwt = p.nwt;
  t.cluster = p.stride / kStatsWarps;
  t.stride = p.stride;
  t.warps = kStatsWarps;
  t.pipe = 0;
  const KernelSet ks = kernels_for(dtype, t);
  return launch_argmax(ks, t, logits, lengths, ws, out, R, P, Pout, lim_off, gamma, V, p.stride, clear_error, st);
}

}  // namespace specv

using namespace specv;

extern "C" size_t specv_verify_chain_workspace_size(int R, int gamma, int V, specv_dtype dtype) {
  if (R < 0 || gamma < 0 || gamma > SPECV_MAX_GAMMA || V < 1 || (dtype != SPECV_F32 && dtype != SPECV_BF16)) return 0;
  // enough for whichever tiling a call may pick (aligned or unaligned rows)
  size_t need = 0;
  for (int vec = 0; vec < 2; ++vec) {
    if (vec && V % (dtype == SPECV_BF16 ? 8 : 4) != 0) continue;
    Tiling t;
    if (choose_tiling(V, dtype, vec != 0, &t)) {
      const size_t n = chain_layout(R, gamma, t).total;
      if (n > need) need = n;
    }
    if (choose_pipe(V, dtype, vec != 0, &t)) {
      const size_t n = chain_layout(R, gamma, t).total;
      if (n > need) need = n;
    }
  }
  return need;
}

static specv_status validate_temperature(float T) {
  if (!(T >= 0.f) || !isfinite(T) || (T > 0.f && T < kMinTemperature)) return SPECV_ERR_INVALID_ARG;
  return SPECV_OK;
}

extern "C" specv_status specv_verify_chain(const void* target_logits, const void* draft_logits, specv_dtype dtype,
                                           const int32_t* draft_tokens, const int32_t* lengths, const float* uniforms,
                                           int R, int gamma, int V, float temperature, int32_t* accepted_len,
                                           int32_t* out_token, float* c_star, void* workspace, size_t workspace_bytes,
                                           void* stream) {
  if (dtype != SPECV_F32 && dtype != SPECV_BF16) return SPECV_ERR_INVALID_ARG;
  if (R < 0 || gamma < 0 || gamma > SPECV_MAX_GAMMA || V < 1) return SPECV_ERR_INVALID_ARG;
  if (validate_temperature(temperature) != SPECV_OK) return SPECV_ERR_INVALID_ARG;
  if (R == 0) return SPECV_OK;
  const size_t esz = dtype == SPECV_BF16 ? 2 : 4;
  if (!target_logits || !accepted_len || !out_token || !workspace) return SPECV_ERR_INVALID_ARG;
  if (gamma > 0 && !draft_tokens) return SPECV_ERR_INVALID_ARG;
  const bool need_draft = temperature > 0.f || c_star != nullptr;
  if (need_draft && gamma > 0 && !draft_logits) return SPECV_ERR_INVALID_ARG;
  if (temperature > 0.f && !uniforms) return SPECV_ERR_INVALID_ARG;
  if (!aligned_to(target_logits, esz) || !aligned_to(draft_logits, esz) || !aligned_to(draft_tokens, 4) ||
      !aligned_to(lengths, 4) || !aligned_to(uniforms, 4) || !aligned_to(accepted_len, 4) ||
      !aligned_to(out_token, 4) || !aligned_to(c_star, 4) || !aligned_to(workspace, 256))
    return SPECV_ERR_INVALID_ARG;
  const bool vec_ok = rows_vector_ok(target_logits, V, dtype) && rows_vector_ok(draft_logits, V, dtype);
  Tiling t;
  if (temperature > 0.f ? !choose_sampling_tiling(V, dtype, vec_ok, &t) : !choose_tiling(V, dtype, vec_ok, &t))
    return SPECV_ERR_UNSUPPORTED;
  if (workspace_bytes < chain_layout(R, gamma, t).total) return SPECV_ERR_INVALID_ARG;
  specv_status s = check_device();
  if (s != SPECV_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (temperature > 0.f)
    return chain_sampling(target_logits, draft_logits, dtype, draft_tokens, lengths, uniforms, R, gamma, gamma + 1,
                          gamma + 1, gamma, V, temperature, accepted_len, out_token, c_star, workspace, t, st, true);
  return chain_greedy(target_logits, draft_logits, dtype, draft_tokens, lengths, R, gamma, gamma + 1, V, accepted_len,
                      out_token, c_star, workspace, t, st, true);
}

extern "C" size_t specv_tv_accept_workspace_size(int R, int gamma, int V, specv_dtype dtype) {
  return specv_verify_chain_workspace_size(R, gamma, V, dtype);
}

extern "C" specv_status specv_tv_accept(const void* target_logits, const void* draft_logits, specv_dtype dtype, int R,
                                        int gamma, int target_positions, int V, float temperature, float* c_star,
                                        void* workspace, size_t workspace_bytes, void* stream) {
  if (dtype != SPECV_F32 && dtype != SPECV_BF16) return SPECV_ERR_INVALID_ARG;
  if (R < 0 || gamma < 0 || gamma > SPECV_MAX_GAMMA || V < 1 || target_positions < gamma) return SPECV_ERR_INVALID_ARG;
  if (validate_temperature(temperature) != SPECV_OK) return SPECV_ERR_INVALID_ARG;
  if (R == 0 || gamma == 0) return SPECV_OK;
  const size_t esz = dtype == SPECV_BF16 ? 2 : 4;
  if (!target_logits || !draft_logits || !c_star || !workspace) return SPECV_ERR_INVALID_ARG;
  if (!aligned_to(target_logits, esz) || !aligned_to(draft_logits, esz) || !aligned_to(c_star, 4) ||
      !aligned_to(workspace, 256))
    return SPECV_ERR_INVALID_ARG;
  const bool vec_ok = rows_vector_ok(target_logits, V, dtype) && rows_vector_ok(draft_logits, V, dtype);
  Tiling t;
  if (temperature > 0.f ? !choose_sampling_tiling(V, dtype, vec_ok, &t) : !choose_tiling(V, dtype, vec_ok, &t))
    return SPECV_ERR_UNSUPPORTED;
  if (workspace_bytes < chain_layout(R, gamma, t).total) return SPECV_ERR_INVALID_ARG;
  specv_status s = check_device();
  if (s != SPECV_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (temperature > 0.f)
    return chain_sampling(target_logits, draft_logits, dtype, nullptr, nullptr, nullptr, R, gamma, gamma,
                          target_positions, gamma, V, temperature, nullptr, nullptr, c_star, workspace, t, st, false);
  return chain_greedy(target_logits, draft_logits, dtype, nullptr, nullptr, R, gamma, target_positions, V, nullptr,
                      nullptr, c_star, workspace, t, st, false);
}
