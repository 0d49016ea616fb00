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

namespace specv {

constexpr int kStatsWarps = 8;        // warps (tiles) per CTA in chain_stats
constexpr int kMaxCluster = 16;
constexpr int kMaxTiles = kStatsWarps * kMaxCluster;   // 128 tiles per row
constexpr int kFinishThreads = 128;
constexpr int kArgmaxWarps = 8;

struct RowRec {
  RowStats s;
  float thr;        // min(1, q(x)/p(x)); NaN if the draft token is out of range
  float pad[3];
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
template <typename Elem, bool VEC, int VPT>
__global__ void __launch_bounds__(kStatsWarps * 32, 2) chain_stats_kernel(StatsArgs a) {
  using S = Slot<Elem, VEC>;
  constexpr int VW = S::VW;
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
  const int tile = int(rank) * kStatsWarps + warp;
  const bool active = tile < a.nwt;

  // the draft token's logits for the accept test, fetched early
  float lq_x = 0.f, lp_x = 0.f;
  bool x_ok = false;
  if (pair && a.tokens && rank == 0 && threadIdx.x == 0) {
    const int x = a.tokens[size_t(r) * a.gamma + k];
    x_ok = x >= 0 && x < a.V;
    if (x_ok) {
      if constexpr (sizeof(Elem) == 2) {
        lq_x = __uint_as_float(uint32_t(__ldg(reinterpret_cast<const unsigned short*>(trow) + x)) << 16);
        lp_x = __uint_as_float(uint32_t(__ldg(reinterpret_cast<const unsigned short*>(drow) + x)) << 16);
      } else {
        lq_x = __ldg(reinterpret_cast<const float*>(trow) + x);
        lp_x = __ldg(reinterpret_cast<const float*>(drow) + x);
      }
    }
  }

  S tq[VPT], tp[VPT];
  if (active) {
#pragma unroll
    for (int j = 0; j < VPT; ++j) tq[j].load(trow, slot_index<VPT, VW>(tile, j, lane), a.V);
    if (pair) {
#pragma unroll
      for (int j = 0; j < VPT; ++j) tp[j].load(drow, slot_index<VPT, VW>(tile, j, lane), a.V);
    }
  }

  // ---- pass 1: tile max and tile normaliser (ex2 domain)
  const float c2 = a.c2;
  float mq = neg_inf(), mp = neg_inf();
  if (active) {
#pragma unroll
    for (int j = 0; j < VPT; ++j) mq = fmaxf(mq, tq[j].vmax());
    if (pair) {
#pragma unroll
      for (int j = 0; j < VPT; ++j) mp = fmaxf(mp, tp[j].vmax());
    }
  }
  mq = warp_max(mq);
  mp = warp_max(mp);
  const bool q_live = mq > neg_inf();
  const bool p_live = mp > neg_inf();
  const float mq_c2 = q_live ? mq * c2 : neg_inf();
  const float mp_c2 = p_live ? mp * c2 : neg_inf();
  float zq = 0.f, zp = 0.f;
  if (q_live) {
#pragma unroll
    for (int j = 0; j < VPT; ++j)
#pragma unroll
      for (int e = 0; e < VW; ++e) zq += ex2(fmaf(tq[j].get(e), c2, -mq_c2));
  }
  if (p_live) {
#pragma unroll
    for (int j = 0; j < VPT; ++j)
#pragma unroll
      for (int e = 0; e < VW; ++e) zp += ex2(fmaf(tp[j].get(e), c2, -mp_c2));
  }
  zq = warp_sum(zq);
  zp = warp_sum(zp);

  // ---- cluster exchange of tile partials
  __shared__ float4 s_tiles[kStatsWarps];
  __shared__ float4 s_row;
  if (lane == 0) s_tiles[warp] = make_float4(mq_c2, zq, mp_c2, zp);
  cluster_arrive_release();
  cluster_wait_acquire();
  if (warp == 0) {
    const int ntile = int(C) * kStatsWarps;
    float4 t[kMaxTiles / 32];
    float Mq = neg_inf(), Mp = neg_inf();
#pragma unroll
    for (int i = 0; i < kMaxTiles / 32; ++i) {
      const int tt = lane + 32 * i;
      if (tt < ntile) {
        t[i] = ld_shared_cluster_f4(cluster_map_shared(&s_tiles[tt % kStatsWarps], uint32_t(tt / kStatsWarps)));
      } else {
        t[i] = make_float4(neg_inf(), 0.f, neg_inf(), 0.f);
      }
      Mq = fmaxf(Mq, t[i].x);
      Mp = fmaxf(Mp, t[i].z);
    }
    Mq = warp_max(Mq);
    Mp = warp_max(Mp);
    float Zq = 0.f, Zp = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxTiles / 32; ++i) {
      if (t[i].y > 0.f) Zq += t[i].y * ex2(t[i].x - Mq);
      if (t[i].w > 0.f) Zp += t[i].w * ex2(t[i].z - Mp);
    }
    Zq = warp_sum(Zq);
    Zp = warp_sum(Zp);
    if (lane == 0) s_row = make_float4(Mq, Zq, Mp, Zp);
  }
  cluster_arrive_relaxed();            // remote shared-memory reads of this CTA are done
  __syncthreads();
  const float4 row = s_row;

  // ---- pass 2: tile residual mass and q mass
  const float sq = q_live ? tile_scale(mq_c2, row.x, row.y) : 0.f;
  const float sp = p_live ? tile_scale(mp_c2, row.z, row.w) : 0.f;
  float resid = 0.f;
  if (pair && q_live) {
#pragma unroll
    for (int j = 0; j < VPT; ++j)
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        const float eq = ex2(fmaf(tq[j].get(e), c2, -mq_c2));
        const float ep = p_live ? ex2(fmaf(tp[j].get(e), c2, -mp_c2)) : 0.f;
        resid += fmaxf(fmaf(eq, sq, -__fmul_rn(ep, sp)), 0.f);
      }
  }
  resid = warp_sum(resid);
  if (lane == 0 && active) {
    TileStats ts;
    ts.mq_c2 = mq_c2;
    ts.mp_c2 = mp_c2;
    ts.resid = resid;
    ts.qmass = __fmul_rn(sq, zq);
    a.tiles[size_t(item) * a.ntile_stride + tile] = ts;
  }
  if (rank == 0 && threadIdx.x == 0) {
    RowRec rr;
    rr.s.Mq_c2 = row.x; rr.s.Zq = row.y; rr.s.Mp_c2 = row.z; rr.s.Zp = row.w;
    rr.thr = __int_as_float(0x7fc00000);
    if (pair && a.tokens && x_ok) {
      const float qx = ex2(fmaf(lq_x, c2, -row.x)) / row.y;
      const float px = ex2(fmaf(lp_x, c2, -row.z)) / row.w;
      rr.thr = px > 0.f ? fminf(1.f, qx / px) : 1.f;
    }
    rr.pad[0] = rr.pad[1] = rr.pad[2] = 0.f;
    a.rows[item] = rr;
  }
  cluster_wait_acquire();              // keep shared memory alive until every CTA has read it
}

// ---------------------------------------------------------------------------
struct FinishArgs {
  const void* target;
  const void* draft;
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

// Inverse-CDF draw inside one tile (one warp).  `use_resid`: weights
// [q - p]_+ (else q).  Returns the first element index v with
// base + C_tile(v) > target, or, if rounding leaves none, the last element with
// positive weight.  Same per-element arithmetic as chain_stats pass 2.
template <typename Elem, bool VEC, int VPT>
__device__ int rescan_tile(const Elem* trow, const Elem* drow, long V, int tile, float c2, const TileStats& ts,
                           const RowStats& rs, bool use_resid, float base, float target) {
  using S = Slot<Elem, VEC>;
  constexpr int VW = S::VW;
  const int lane = threadIdx.x & 31;
  const bool q_live = ts.mq_c2 > neg_inf();
  const bool p_live = use_resid && ts.mp_c2 > neg_inf();
  const float sq = q_live ? tile_scale(ts.mq_c2, rs.Mq_c2, rs.Zq) : 0.f;
  const float sp = p_live ? tile_scale(ts.mp_c2, rs.Mp_c2, rs.Zp) : 0.f;
  float run = base;
  int last_pos = -1;
  for (int j = 0; j < VPT; ++j) {
    const long idx0 = slot_index<VPT, VW>(tile, j, lane);
    S xq, xp;
    xq.load(trow, idx0, V);
    if (use_resid) xp.load(drow, idx0, V);
    float w[VW];
    float lsum = 0.f;
#pragma unroll
    for (int e = 0; e < VW; ++e) {
      float we = 0.f;
      if (q_live) {
        const float eq = ex2(fmaf(xq.get(e), c2, -ts.mq_c2));
        if (use_resid) {
          const float ep = p_live ? ex2(fmaf(xp.get(e), c2, -ts.mp_c2)) : 0.f;
          we = fmaxf(fmaf(eq, sq, -__fmul_rn(ep, sp)), 0.f);
        } else {
          we = __fmul_rn(eq, sq);
        }
      }
      w[e] = we;
      lsum += we;
    }
    const float incl = warp_inclusive_scan(lsum);
    float acc = run + (incl - lsum);
    int cand = 0x7fffffff;
#pragma unroll
    for (int e = 0; e < VW; ++e) {
      acc += w[e];
      if (w[e] > 0.f) last_pos = int(idx0) + e;
      if (cand == 0x7fffffff && acc > target && w[e] > 0.f) cand = int(idx0) + e;
    }
    int best = cand;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = min(best, __shfl_xor_sync(0xffffffffu, best, o));
    if (best != 0x7fffffff) return best;
    run = __shfl_sync(0xffffffffu, acc, 31);
  }
  int lp = last_pos;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
  return lp;
}

template <typename Elem, bool VEC, int VPT>
__global__ void __launch_bounds__(kFinishThreads) chain_finish_kernel(FinishArgs a) {
  const int r = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gamma = a.gamma;
  int ell = a.lengths ? a.lengths[r] : gamma;
  bool bad = ell < 0 || ell > gamma;
  if (bad) ell = 0;

  // ---- c*_k = 1 - sum of tile residual masses
  if (a.c_star) {
    for (int k = warp; k < gamma; k += kFinishThreads / 32) {
      float c = __int_as_float(0x7fc00000);
      if (!bad && k < ell) {
        const TileStats* ts = a.tiles + size_t(r * a.P + k) * a.ntile_stride;
        float s = 0.f;
        for (int t = lane; t < a.nwt; t += 32) s += ts[t].resid;
        s = warp_sum(s);
        c = 1.f - s;
      }
      if (lane == 0) a.c_star[size_t(r) * gamma + k] = c;
    }
  }
  if (!a.sample || warp != 0) return;

  // ---- first rejection (warp ballot over the accept tests)
  bool acc_ok = true, valid = true;
  if (lane < ell) {
    const float thr = a.rows[r * a.P + lane].thr;
    const float u0 = a.uniforms[(size_t(r) * (gamma + 1) + lane) * 2];
    valid = !isnan(thr) && u0 >= 0.f && u0 < 1.f;
    acc_ok = u0 < thr;
  }
  bad = bad || __any_sync(0xffffffffu, !valid);
  const unsigned rej = __ballot_sync(0xffffffffu, !acc_ok) & (ell >= 32 ? 0xffffffffu : ((1u << ell) - 1u));
  const int A = rej ? __ffs(rej) - 1 : ell;
  const float u1 = a.uniforms[(size_t(r) * (gamma + 1) + A) * 2 + 1];
  bad = bad || !(u1 >= 0.f && u1 < 1.f);
  if (bad) {
    if (lane == 0) {
      a.accepted[r] = -1;
      a.out_token[r] = -1;
      record_device_error(a.workspace, SPECV_ERR_DEVICE_DATA);
    }
    return;
  }

  // ---- inverse-CDF draw: residual of position A (rejection) or q at l_r (bonus)
  const int item = r * a.P + A;
  const TileStats* ts = a.tiles + size_t(item) * a.ntile_stride;
  const RowStats rs = a.rows[item].s;
  bool use_resid = A < ell;
  const int per = (a.nwt + 31) / 32;          // consecutive tiles per lane (index order)
  const int t0 = lane * per, t1 = min(a.nwt, t0 + per);
  float lsum = 0.f;
  for (int t = t0; t < t1; ++t) lsum += use_resid ? ts[t].resid : ts[t].qmass;
  float incl = warp_inclusive_scan(lsum);
  float total = __shfl_sync(0xffffffffu, incl, 31);
  if (use_resid && !(total > 0.f)) {          // no residual mass: draw from q
    use_resid = false;
    lsum = 0.f;
    for (int t = t0; t < t1; ++t) lsum += ts[t].qmass;
    incl = warp_inclusive_scan(lsum);
    total = __shfl_sync(0xffffffffu, incl, 31);
  }
  const float target = u1 * total;
  // the tile holding the target: first lane whose range crosses it, then its tiles in order
  const unsigned hit = __ballot_sync(0xffffffffu, incl > target && t1 > t0);
  int sel_tile = -1;
  float base = 0.f;
  if (hit) {
    const int L = __ffs(hit) - 1;
    if (lane == L) {
      float run = incl - lsum;
      for (int t = t0; t < t1; ++t) {
        const float m = use_resid ? ts[t].resid : ts[t].qmass;
        if (run + m > target && m > 0.f) { sel_tile = t; base = run; break; }
        run += m;
      }
      if (sel_tile < 0) {                     // rounding: take this lane's last tile with mass
        run = incl - lsum;
        for (int t = t0; t < t1; ++t) {
          const float m = use_resid ? ts[t].resid : ts[t].qmass;
          if (m > 0.f) { sel_tile = t; base = run; }
          run += m;
        }
      }
    }
    sel_tile = __shfl_sync(0xffffffffu, sel_tile, L);
    base = __shfl_sync(0xffffffffu, base, L);
  }
  if (sel_tile < 0) {                          // rounding at the top: last tile with mass
    int cand = -1;
    for (int t = t0; t < t1; ++t)
      if ((use_resid ? ts[t].resid : ts[t].qmass) > 0.f) cand = t;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cand = max(cand, __shfl_xor_sync(0xffffffffu, cand, o));
    sel_tile = cand;
    base = 0.f;
    // prefix before cand
    float pre = 0.f;
    for (int t = t0; t < t1; ++t)
      if (t < cand) pre += use_resid ? ts[t].resid : ts[t].qmass;
    base = warp_sum(pre);
  }
  int tok = -1;
  if (sel_tile >= 0) {
    const Elem* trow = reinterpret_cast<const Elem*>(a.target) + (size_t(r) * a.Pt + A) * a.V;
    const Elem* drow = use_resid ? reinterpret_cast<const Elem*>(a.draft) + (size_t(r) * a.Pd + A) * a.V : nullptr;
    tok = rescan_tile<Elem, VEC, VPT>(trow, drow, a.V, sel_tile, a.c2, ts[sel_tile], rs, use_resid, base, target);
  }
  if (lane == 0) {
    a.accepted[r] = A;
    a.out_token[r] = tok;
    if (tok < 0) record_device_error(a.workspace, SPECV_ERR_DEVICE_DATA);
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

__global__ void __launch_bounds__(32) greedy_finish_kernel(GreedyArgs a) {
  const int r = blockIdx.x;
  const int lane = threadIdx.x;
  const int gamma = a.gamma;
  int ell = a.lengths ? a.lengths[r] : gamma;
  bool bad = ell < 0 || ell > gamma;
  if (bad) ell = 0;
  // g_k and the draft argmax for k < ell: lane k keeps row k (gamma <= 32)
  int my_g = -1, my_gd = -1;
  for (int k = 0; k < ell; ++k) {
    const int g = combine_argmax(a.targ + size_t(r * a.tpos + k) * a.ntile_stride, a.nwt);
    if (lane == k) my_g = g;
    if (a.darg) {
      const int gd = combine_argmax(a.darg + size_t(r * gamma + k) * a.ntile_stride, a.nwt);
      if (lane == k) my_gd = gd;
    }
  }
  if (a.c_star) {
    for (int k = lane; k < gamma; k += 32) {
      float c = __int_as_float(0x7fc00000);
      if (!bad && k < ell) c = (my_gd == my_g) ? 1.f : 0.f;
      a.c_star[size_t(r) * gamma + k] = c;
    }
  }
  if (!a.sample) return;
  bool mismatch = false, valid = true;
  if (lane < ell) {
    const int x = a.tokens[size_t(r) * gamma + lane];
    valid = x >= 0 && x < a.V;
    mismatch = x != my_g;
  }
  bad = bad || __any_sync(0xffffffffu, !valid);
  const unsigned mm = __ballot_sync(0xffffffffu, mismatch);
  const int A = mm ? __ffs(mm) - 1 : ell;
  // correction (A < l_r) or bonus (A = l_r) token: the target argmax of row A
  const int tok = combine_argmax(a.targ + size_t(r * a.tpos + A) * a.ntile_stride, a.nwt);
  if (lane == 0) {
    a.accepted[r] = bad ? -1 : A;
    a.out_token[r] = bad ? -1 : tok;
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
};

constexpr int kVptList[] = {1, 2, 4, 6, 8, 10};

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
        return true;
      }
    }
  }
  return false;
}

template <typename Elem, bool VEC, int VPT>
struct ChainKernels {
  static void* stats() { return reinterpret_cast<void*>(&chain_stats_kernel<Elem, VEC, VPT>); }
  static void* finish() { return reinterpret_cast<void*>(&chain_finish_kernel<Elem, VEC, VPT>); }
  static void* argmax() { return reinterpret_cast<void*>(&argmax_tiles_kernel<Elem, VEC, VPT>); }
};

struct KernelSet {
  void* stats;
  void* finish;
  void* argmax;
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

KernelSet kernels_for(specv_dtype dtype, const Tiling& t) {
  if (dtype == SPECV_BF16) return t.vec ? pick_vpt<uint16_t, true>(t.vpt) : pick_vpt<uint16_t, false>(t.vpt);
  return t.vec ? pick_vpt<float, true>(t.vpt) : pick_vpt<float, false>(t.vpt);
}

// Workspace: header | rows RowRec[items] | tiles TileStats[items][ntile_stride]
//            | target argmax ArgRec[R*(gamma+1)][stride] | draft argmax ArgRec[R*gamma][stride]
struct ChainLayout {
  size_t rows_off, tiles_off, targ_off, darg_off, total;
  int ntile_stride;
};

ChainLayout chain_layout(int R, int gamma, const Tiling& t) {
  ChainLayout L;
  L.ntile_stride = t.cluster * kStatsWarps;
  const size_t items = size_t(R) * (gamma + 1);
  size_t off = kHeaderBytes;
  L.rows_off = off;
  off = align256(off + items * sizeof(RowRec));
  L.tiles_off = off;
  off = align256(off + items * L.ntile_stride * sizeof(TileStats));
  L.targ_off = off;
  off = align256(off + items * L.ntile_stride * sizeof(ArgRec));
  L.darg_off = off;
  off = align256(off + size_t(R) * gamma * L.ntile_stride * sizeof(ArgRec));
  L.total = off;
  return L;
}

bool rows_vector_ok(const void* p, long V, specv_dtype dtype) {
  const int vw = dtype == SPECV_BF16 ? 8 : 4;
  return p == nullptr || ((reinterpret_cast<uintptr_t>(p) & 15) == 0 && V % vw == 0);
}

specv_status launch_stats(const KernelSet& ks, const Tiling& t, const StatsArgs& sa, int items, cudaStream_t st) {
  if (items == 0) return SPECV_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(items) * unsigned(t.cluster));
  cfg.blockDim = dim3(kStatsWarps * 32);
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
  specv_status s = launch_stats(ks, t, sa, R * P, st);
  if (s != SPECV_OK) return s;
  FinishArgs fa;
  fa.target = target;
  fa.draft = draft;
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
  if (cudaLaunchKernel(ks.finish, dim3(R), dim3(kFinishThreads), fargs, 0, st) != cudaSuccess) return SPECV_ERR_CUDA;
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
  if (cudaLaunchKernel(reinterpret_cast<void*>(&greedy_finish_kernel), dim3(R), dim3(32), gargs, 0, st) != cudaSuccess)
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
    Tiling t;
    if (vec && V % (dtype == SPECV_BF16 ? 8 : 4) != 0) continue;
    if (choose_tiling(V, dtype, vec != 0, &t)) {
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
  if (!choose_tiling(V, dtype, vec_ok, &t)) return SPECV_ERR_UNSUPPORTED;
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
  if (!choose_tiling(V, dtype, vec_ok, &t)) return SPECV_ERR_UNSUPPORTED;
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
