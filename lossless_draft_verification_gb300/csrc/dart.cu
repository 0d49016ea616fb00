// DART's candidate-tree construction without the n-gram index (sm_103a).
//
// Method (DART reading notes §5.2-5.3, Algorithm 3 steps 1-8, with the n-gram
// score g == 1): for each future offset i = 1..d the top-k tokens of the draft
// softmax p_i; active paths start at the root with score 0; every active path
// is extended by every top-k token with eq. (10)'s increment
//   ds = (0.9^i log(p_i(v) + eps) + 0.5 log(1 + eps)) / (i + 1)^0.7,
// every extension joins the node set T and the w best become the next active
// paths; then theta nodes are selected and handed to the verifier as a tree.
//
// Kernels
//   dart_topk_tiles  one warp per (row, warp tile) of the [R, d, V] draft
//                    logits: the tile's softmax partial (max * c2, sum of
//                    2^(x c2 - max c2)) and its top-k (logit, id) candidates by
//                    repeated warp argmax (lowest id among equal logits).  The
//                    only pass over the logits: HBM-bound.
//   dart_build       one CTA per request: warp i merges offset i's tile
//                    candidates into the top-k and forms log p(v) in float64
//                    from the combined normaliser; the beam over depths ranks
//                    its w * k candidates by counting (score, then generation
//                    order); the selection takes, theta times, the best node of
//                    the frontier (children of the nodes taken so far) by the
//                    key min(score, parent key), then smaller depth, then
//                    generation order -- since keys never increase along a path
//                    and equal keys go to the shallower node, this is the theta
//                    largest keys of T, ancestor-closed; thread 0 then writes
//                    the tree depth-first (children in selection order).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "host_common.h"

namespace specv {

constexpr int kDartTileWarps = 8;
constexpr int kDartBuildThreads = 256;
constexpr int kDartMaxK = 32;
constexpr int kDartMaxW = 32;
constexpr int kDartMaxDepth = 8;            // one warp per offset in dart_build
constexpr int kDartMaxTheta = 1023;
constexpr int kDartVpt = 10;                // slots per lane and row in dart_topk_tiles
constexpr int kDartMaxTilesPerLane = 4;     // warp tiles per row <= 128

struct DartCand {
  float v;                                  // logit (raw, before 1/T)
  int i;                                    // token id
};

struct DartTileArgs {
  const void* logits;                       // [R, d, V]
  float2* part;                             // [R * d, ntile]: (max * c2, Z)
  DartCand* cand;                           // [R * d, ntile, k]
  long V;
  int rows, ntile, k;
  float c2;
};

template <typename Elem>
__global__ void __launch_bounds__(kDartTileWarps * 32) dart_topk_tiles_kernel(DartTileArgs a) {
  using S = Slot<Elem, true>;
  constexpr int VW = S::VW;
  const int lane = threadIdx.x & 31;
  const long unit = long(blockIdx.x) * kDartTileWarps + (threadIdx.x >> 5);
  if (unit >= long(a.rows) * a.ntile) return;
  const int row = int(unit / a.ntile), tile = int(unit - long(row) * a.ntile);
  const Elem* x = reinterpret_cast<const Elem*>(a.logits) + size_t(row) * size_t(a.V);
  float val[kDartVpt * VW];
#pragma unroll
  for (int j = 0; j < kDartVpt; ++j) {
    S s;
    s.load(x, slot_index<kDartVpt, VW>(tile, j, lane), a.V);
#pragma unroll
    for (int e = 0; e < VW; ++e) val[j * VW + e] = s.get(e);
  }
  // softmax partial of the tile
  float m = neg_inf();
#pragma unroll
  for (int q = 0; q < kDartVpt * VW; ++q) m = fmaxf(m, val[q]);
  m = warp_max(m);
  float z = 0.f;
  if (m > neg_inf()) {
#pragma unroll
    for (int q = 0; q < kDartVpt * VW; ++q) z += ex2(fmaf(val[q], a.c2, -m * a.c2));
  }
  z = warp_sum(z);
  if (lane == 0) a.part[unit] = make_float2(m > neg_inf() ? m * a.c2 : neg_inf(), z);
  // top-k by repeated argmax; the winning element is struck out
  for (int t = 0; t < a.k; ++t) {
    float bv = neg_inf();
    int bi = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < kDartVpt; ++j)
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        const int id = int(slot_index<kDartVpt, VW>(tile, j, lane)) + e;
        const float v = val[j * VW + e];
        if (id < a.V && (v > bv || (v == bv && id < bi))) { bv = v; bi = id; }
      }
    warp_argmax(bv, bi);
#pragma unroll
    for (int j = 0; j < kDartVpt; ++j)
#pragma unroll
      for (int e = 0; e < VW; ++e)
        if (int(slot_index<kDartVpt, VW>(tile, j, lane)) + e == bi) val[j * VW + e] = neg_inf();
    if (lane == 0) {
      DartCand c;
      c.v = bi == 0x7fffffff ? neg_inf() : bv;
      c.i = bi;
      a.cand[size_t(unit) * a.k + t] = c;
    }
  }
}

struct DartBuildArgs {
  const float2* part;
  const DartCand* cand;
  int32_t* parents;                         // [R, theta + 1]
  int32_t* tokens;                          // [R, theta + 1]
  int32_t* n_nodes;                         // [R]
  void* workspace;
  int d, ntile, k, w, theta;
  double c2;                                // log2(e) / T
  double eps;
};

// node of T in shared memory; its index is its generation order
struct DartNode {
  double score;
  unsigned long long s_ord, k_ord;          // order-preserving integer images of score and key
  int parent;                               // node index, -1 for the root
  int token;
  int depth;
  int child0;                               // first of its k children in T, -1 if never extended
};

// An unsigned integer with the order of the double x (x not NaN): comparisons
// then run on the integer units, not on the narrow float64 pipe.
__device__ __forceinline__ unsigned long long dart_ord(double x) {
  const unsigned long long u = static_cast<unsigned long long>(__double_as_longlong(x));
  return (u >> 63) ? ~u : (u | (1ull << 63));
}

// (key, depth, generation order): larger key first, then shallower, then older
__device__ __forceinline__ bool dart_better(unsigned long long ka, int da, int ia, unsigned long long kb, int db,
                                            int ib) {
  return ka > kb || (ka == kb && (da < db || (da == db && ia < ib)));
}

__global__ void __launch_bounds__(kDartBuildThreads) dart_build_kernel(DartBuildArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  DartNode* T = reinterpret_cast<DartNode*>(smem);                 // [k + (d - 1) w k]
  __shared__ int s_tok[kDartMaxDepth][kDartMaxK];
  __shared__ double s_lp[kDartMaxDepth][kDartMaxK];
  __shared__ int s_active[kDartMaxW];
  __shared__ int s_sel[kDartMaxTheta];
  __shared__ int s_lbase[kDartMaxTheta + 1], s_lhead[kDartMaxTheta + 1];
  __shared__ int s_nlist;
  const int r = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d = a.d, k = a.k, w = a.w;
  if (r == 0 && tid == 0) *reinterpret_cast<int*>(a.workspace) = 0;

  // ---- per offset (one warp each): the normaliser in float64 and the top-k of
  // the tile candidates, with ln(p(v) + eps) of each pick
  for (int i = warp; i < d; i += kDartBuildThreads / 32) {
    const size_t row = size_t(r) * d + i;
    const float2* pt = a.part + row * a.ntile;
    float M = neg_inf();
    for (int t = lane; t < a.ntile; t += 32) M = fmaxf(M, pt[t].x);
    M = warp_max(M);
    double Z = 0.0;
    for (int t = lane; t < a.ntile; t += 32)
      if (pt[t].y > 0.f) Z += double(pt[t].y) * exp2(double(pt[t].x) - double(M));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, o);
    const double lse2 = double(M) + log2(Z);                // log2 of sum_v 2^(x_v c2)
    // k-way merge of the tiles' candidate lists (each in descending order): lane
    // l owns tiles l, l + 32, l + 64, l + 96 and the head index of each
    const DartCand* c = a.cand + row * a.ntile * k;
    int head[kDartMaxTilesPerLane];
    DartCand hc[kDartMaxTilesPerLane];                       // each owned tile's current head
#pragma unroll
    for (int u = 0; u < kDartMaxTilesPerLane; ++u) {
      head[u] = 0;
      const int tile = lane + 32 * u;
      hc[u] = tile < a.ntile ? c[size_t(tile) * k] : DartCand{neg_inf(), 0x7fffffff};
    }
    float px = 0.f;                                          // lane t: logit of pick t
    for (int t = 0; t < k; ++t) {
      float bv = neg_inf();
      int bi = 0x7fffffff, bu = -1;
#pragma unroll
      for (int u = 0; u < kDartMaxTilesPerLane; ++u) {
        const DartCand x = hc[u];
        if (x.i != 0x7fffffff && (x.v > bv || (x.v == bv && x.i < bi))) { bv = x.v; bi = x.i; bu = u; }
      }
      const int mine = bi;
      warp_argmax(bv, bi);                      // all lanes take part
      if (bi != 0x7fffffff && mine == bi) {     // the owner of the pick advances that tile
#pragma unroll
        for (int u = 0; u < kDartMaxTilesPerLane; ++u)
          if (u == bu) {
            ++head[u];
            hc[u] = head[u] < k ? c[size_t(lane + 32 * u) * k + head[u]] : DartCand{neg_inf(), 0x7fffffff};
          }
      }
      if (lane == t) px = bv;
      if (lane == 0) s_tok[i][t] = bi;
    }
    __syncwarp();
    if (lane < k) {                             // ln(p + eps) of every pick at once
      const int t = lane;
      const double lp = s_tok[i][t] == 0x7fffffff ? -INFINITY : (double(px) * a.c2 - lse2) * 0.6931471805599453;
      s_lp[i][t] = log(exp(lp) + a.eps);
    }
  }
  __syncthreads();

  __syncthreads();
  if (warp != 0) return;
  // Everything below runs in warp 0: the beam and the selection are merges of
  // lists that are already ordered, so no block barrier is needed.
  //
  // ---- beam over depths.  T[0 .. k) are the root's children; at depth i >= 2
  // active path j's k extensions are T[nb + j k .. + k).  A path's extensions
  // come in the order of its offset's picks, i.e. by non-increasing score, so
  // the w best of a depth are a w-way merge of those lists (lane j owns list j).
  const double ng = 0.5 * log(1.0 + a.eps);
  {
    const double sc1 = pow(2.0, 0.7);
    for (int t = lane; t < k; t += 32) {
      const double sv = (0.9 * s_lp[0][t] + ng) / sc1;
      DartNode n;
      n.score = sv;
      n.s_ord = dart_ord(sv);
      n.k_ord = n.s_ord;
      n.parent = -1;
      n.token = s_tok[0][t];
      n.depth = 1;
      n.child0 = -1;
      T[t] = n;
    }
  }
  int nact = min(w, k);
  for (int j = lane; j < nact; j += 32) s_active[j] = j;
  __syncwarp();
  int base = 0, count = k;
  for (int i = 2; i <= d; ++i) {
    const int nb = base + count;
    const double pw = pow(0.9, double(i)), sc = pow(double(i + 1), 0.7);
    for (int q = lane; q < nact * k; q += 32) {
      const int j = q / k, t = q - j * k;
      const DartNode& par = T[s_active[j]];
      DartNode n;
      n.score = par.score + (pw * s_lp[i - 1][t] + ng) / sc;
      n.s_ord = dart_ord(n.score);
      n.k_ord = n.s_ord < par.k_ord ? n.s_ord : par.k_ord;     // key = min(score, parent key)
      n.parent = s_active[j];
      n.token = s_tok[i - 1][t];
      n.depth = i;
      n.child0 = -1;
      T[nb + q] = n;
    }
    for (int j = lane; j < nact; j += 32) T[s_active[j]].child0 = nb + j * k;
    __syncwarp();
    const int nnext = min(w, nact * k);
    int h = 0;                                                 // lane j: head of list j
    int pick = -1;
    for (int p = 0; p < nnext; ++p) {
      unsigned long long bo = 0;
      int bg = 0x7fffffff;
      if (lane < nact && h < k) { bg = nb + lane * k + h; bo = T[bg].s_ord; }
      unsigned long long wo = bo;
      int wg = bg;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long oo = __shfl_xor_sync(0xffffffffu, wo, o);
        const int og = __shfl_xor_sync(0xffffffffu, wg, o);
        if (oo > wo || (oo == wo && og < wg)) { wo = oo; wg = og; }
      }
      if (wg == bg) ++h;                                       // the winning list advances
      if (lane == p) pick = wg;
    }
    if (lane < nnext) s_active[lane] = pick;               // nnext <= w <= 32: lane p holds pick p
    __syncwarp();
    base = nb;
    count = nact * k;
    nact = nnext;
  }
  const int total = base + count;

  // ---- best-first selection: a merge of the open child lists.  The root's
  // list is T[0 .. k); a picked node that was extended opens its k children.
  // Within a list keys do not increase, and across lists the order is (key
  // desc, depth asc, generation asc), so every pick is the best node left.
  const int want = min(a.theta, total);
  if (lane == 0) { s_lbase[0] = 0; s_lhead[0] = 0; s_nlist = 1; }
  __syncwarp();
  for (int p = 0; p < want; ++p) {
    const int nl = s_nlist;
    unsigned long long bk = 0;
    int bd = 0x7fffffff, bi = 0x7fffffff, bl = -1;
    for (int l = lane; l < nl; l += 32) {
      if (s_lhead[l] >= k) continue;
      const int id = s_lbase[l] + s_lhead[l];
      const DartNode& n = T[id];
      if (bl < 0 || dart_better(n.k_ord, n.depth, id, bk, bd, bi)) { bk = n.k_ord; bd = n.depth; bi = id; bl = l; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long ok = __shfl_xor_sync(0xffffffffu, bk, o);
      const int od = __shfl_xor_sync(0xffffffffu, bd, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const int ol = __shfl_xor_sync(0xffffffffu, bl, o);
      if (ol >= 0 && (bl < 0 || dart_better(ok, od, oi, bk, bd, bi))) { bk = ok; bd = od; bi = oi; bl = ol; }
    }
    if (lane == 0) {
      s_sel[p] = bi;
      ++s_lhead[bl];
      const int c0 = T[bi].child0;
      if (c0 >= 0) {
        s_lbase[s_nlist] = c0;
        s_lhead[s_nlist] = 0;
        ++s_nlist;
      }
    }
    __syncwarp();
  }

  // ---- the tree, depth first from the root, children in selection order.
  // Child lists first (selection order kept), then one walk; T[].depth and
  // T[].child0 are reused as the next-sibling link and the output row.
  if (tid == 0) {
    int32_t* par_out = a.parents + size_t(r) * (a.theta + 1);
    int32_t* tok_out = a.tokens + size_t(r) * (a.theta + 1);
    for (int q = 0; q <= a.theta; ++q) { par_out[q] = -1; tok_out[q] = 0; }
    int root_first = -1, root_last = -1;
    for (int q = 0; q < want; ++q) {                  // first / last child of each selected node
      T[s_sel[q]].score = __longlong_as_double(-1ll); // first child (as an int in the bits)
      T[s_sel[q]].s_ord = ~0ull;                       // last child
    }
    for (int q = 0; q < want; ++q) {
      const int id = s_sel[q];
      T[id].depth = -1;                               // next sibling
      const int pa = T[id].parent;
      if (pa < 0) {
        if (root_first < 0) root_first = id; else T[root_last].depth = id;
        root_last = id;
      } else {
        const int last = int(static_cast<long long>(T[pa].s_ord));
        if (last < 0) T[pa].score = __longlong_as_double(id); else T[last].depth = id;
        T[pa].s_ord = static_cast<unsigned long long>(static_cast<long long>(id));
      }
    }
    int next = 1;
    int stack[kDartMaxDepth + 1];
    int sp = -1;
    for (int id = root_first; id >= 0;) {
      T[id].child0 = next;
      const int pa = T[id].parent;
      par_out[next] = pa < 0 ? 0 : T[pa].child0;
      tok_out[next] = T[id].token;
      ++next;
      const int first = int(__double_as_longlong(T[id].score));
      if (first >= 0) {                               // descend
        stack[++sp] = id;
        id = first;
        continue;
      }
      int sib = T[id].depth;                          // else the next sibling, climbing as needed
      while (sib < 0 && sp >= 0) sib = T[stack[sp--]].depth;
      id = sib;
    }
    a.n_nodes[r] = next;
  }
}

}  // namespace specv

using namespace specv;

namespace {
constexpr double kDartEps = 1e-10;

struct DartPlan {
  int vw, ntile;
  size_t part_off, cand_off, total;
  size_t build_smem;
};

bool dart_plan(int R, int d, long V, int k, int w, int theta, specv_dtype dtype, DartPlan* p) {
  p->vw = dtype == SPECV_BF16 ? 8 : 4;
  const long tile = 32L * kDartVpt * p->vw;
  const long ntile = (V + tile - 1) / tile;
  if (ntile > 32L * kDartMaxTilesPerLane) return false;
  p->ntile = int(ntile);
  const size_t rows = size_t(R) * d;
  size_t off = kHeaderBytes;
  p->part_off = off;
  off = align256(off + rows * ntile * sizeof(float2));
  p->cand_off = off;
  off = align256(off + rows * ntile * k * sizeof(DartCand));
  p->total = off;
  const size_t nodes = size_t(k) + size_t(d - 1) * w * k;
  p->build_smem = nodes * sizeof(DartNode) + (size_t(k) + size_t(theta) * k) * sizeof(int);
  return p->build_smem <= 200 * 1024;
}

bool dart_args_ok(int R, int d, int V, int k, int w, int theta, specv_dtype dtype) {
  return R >= 0 && d >= 1 && d <= kDartMaxDepth && V >= 1 && k >= 1 && k <= kDartMaxK && k <= V && w >= 1 &&
         w <= kDartMaxW && theta >= 1 && theta <= kDartMaxTheta && (dtype == SPECV_F32 || dtype == SPECV_BF16);
}
}  // namespace

extern "C" size_t specv_dart_tree_workspace_size(int R, int d, int V, int k, int w, int theta, specv_dtype dtype) {
  if (!dart_args_ok(R, d, V, k, w, theta, dtype)) return 0;
  DartPlan p;
  if (!dart_plan(R, d, V, k, w, theta, dtype, &p)) return 0;
  return p.total;
}

extern "C" specv_status specv_dart_tree(const void* draft_logits, specv_dtype dtype, int R, int d, int V,
                                        float temperature, int k, int w, int theta, int32_t* parents,
                                        int32_t* tokens, int32_t* n_nodes, void* workspace, size_t workspace_bytes,
                                        void* stream) {
  if (!dart_args_ok(R, d, V, k, w, theta, dtype)) return SPECV_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !isfinite(temperature)) return SPECV_ERR_INVALID_ARG;
  if (R == 0) return SPECV_OK;
  if (!draft_logits || !parents || !tokens || !n_nodes || !workspace) return SPECV_ERR_INVALID_ARG;
  const int vw = dtype == SPECV_BF16 ? 8 : 4;
  if (!aligned_to(draft_logits, 16) || V % vw != 0) return SPECV_ERR_UNSUPPORTED;   // 16-byte rows only
  if (!aligned_to(parents, 4) || !aligned_to(tokens, 4) || !aligned_to(n_nodes, 4) || !aligned_to(workspace, 256))
    return SPECV_ERR_INVALID_ARG;
  DartPlan p;
  if (!dart_plan(R, d, V, k, w, theta, dtype, &p)) return SPECV_ERR_UNSUPPORTED;
  if (workspace_bytes < p.total) return SPECV_ERR_INVALID_ARG;
  specv_status s = check_device();
  if (s != SPECV_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  DartTileArgs ta;
  ta.logits = draft_logits;
  ta.part = reinterpret_cast<float2*>(ws + p.part_off);
  ta.cand = reinterpret_cast<DartCand*>(ws + p.cand_off);
  ta.V = V;
  ta.rows = R * d;
  ta.ntile = p.ntile;
  ta.k = k;
  ta.c2 = float(kLog2e / double(temperature));
  void* targs[] = {&ta};
  const long units = long(R) * d * p.ntile;
  const void* tfn = dtype == SPECV_BF16 ? reinterpret_cast<const void*>(&dart_topk_tiles_kernel<uint16_t>)
                                        : reinterpret_cast<const void*>(&dart_topk_tiles_kernel<float>);
  if (cudaLaunchKernel(tfn, dim3(unsigned((units + kDartTileWarps - 1) / kDartTileWarps)), dim3(kDartTileWarps * 32),
                       targs, 0, st) != cudaSuccess)
    return SPECV_ERR_CUDA;
  DartBuildArgs ba;
  ba.part = ta.part;
  ba.cand = ta.cand;
  ba.parents = parents;
  ba.tokens = tokens;
  ba.n_nodes = n_nodes;
  ba.workspace = workspace;
  ba.d = d;
  ba.ntile = p.ntile;
  ba.k = k;
  ba.w = w;
  ba.theta = theta;
  ba.c2 = double(ta.c2);
  ba.eps = kDartEps;
  if (cudaFuncSetAttribute(reinterpret_cast<const void*>(&dart_build_kernel), cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(p.build_smem)) != cudaSuccess)
    return SPECV_ERR_CUDA;
  void* bargs[] = {&ba};
  if (cudaLaunchKernel(reinterpret_cast<const void*>(&dart_build_kernel), dim3(unsigned(R)), dim3(kDartBuildThreads),
                       bargs, p.build_smem, st) != cudaSuccess)
    return SPECV_ERR_CUDA;
  return SPECV_OK;
}
