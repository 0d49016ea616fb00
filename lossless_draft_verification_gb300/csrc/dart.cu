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
//                    logits, in the only pass over them (HBM-bound): the
//                    tile's softmax partial (max * c2, sum of 2^(x c2 - max c2))
//                    and its top-k (logit, id) candidates, lowest id first
//                    among equal logits.  The k-th largest of the 32 lane
//                    maxima comes from k distinct elements, so it bounds the
//                    tile's k-th best from below: only the few values at or
//                    above it are compacted to shared memory and ranked by
//                    counting.
//   dart_build       one CTA per request: warp i merges offset i's tile lists
//                    into the row's top-k (the same bound, from the lists'
//                    heads), ln(p(v) + eps) from the combined normaliser and
//                    eq. (10)'s increments; all threads
//                    extend the active paths and one warp keeps the w best (a
//                    merge of the score-ordered extension lists); the
//                    selection is a block-wide radix select of the theta
//                    largest keys min(score, parent key), then smaller depth,
//                    then generation order -- keys never increase along a path
//                    and equal keys go to the shallower node, so the theta best
//                    are ancestor-closed; the tree's depth-first rows
//                    (children in selection order) come from subtree sizes,
//                    one barrier per depth.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <cuda_bf16.h>
#include <type_traits>

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
constexpr int kDartMaxTiles = 128;          // warp tiles per row
constexpr int kDartSurvCap = 128;           // survivors of the bound ranked in shared memory
constexpr int kDartNone = 0x7fffffff;       // id of an empty candidate slot

struct DartCand {
  float v;                                  // logit (raw, before 1/T)
  int i;                                    // token id; kDartNone for an empty slot
};

struct DartTileArgs {
  const void* logits;                       // [R, d, V]
  float2* part;                             // [R * d, ntile]: (max * c2, Z)
  DartCand* cand;                           // [R * d, ntile, k]
  long V;
  int rows, ntile, k;
  float c2;                                 // log2(e) / T
};

// (logit descending, id ascending) as one unsigned integer, larger is better;
// 0 is below every element.  -0 is taken as +0, as the float comparison does.
__device__ __forceinline__ unsigned long long dart_key(float v, int id) {
  uint32_t b = __float_as_uint(v);
  b = b == 0x80000000u ? 0u : b;
  const uint32_t o = b ^ (uint32_t(int32_t(b) >> 31) | 0x80000000u);
  return (static_cast<unsigned long long>(o) << 32) | (~static_cast<uint32_t>(id));
}

__device__ __forceinline__ DartCand dart_unkey(unsigned long long key) {
  const uint32_t o = uint32_t(key >> 32);
  const uint32_t b = (o >> 31) ? (o & 0x7fffffffu) : ~o;
  return DartCand{__uint_as_float(b), int(~uint32_t(key))};
}

// the k-th largest (1 <= k <= 32) of the warp's 32 keys
__device__ __forceinline__ unsigned long long warp_kth_largest(unsigned long long key, int k, int lane) {
  int rank = 0;                             // lanes above, equal keys ordered by lane
#pragma unroll
  for (int l = 0; l < 32; ++l) {
    const unsigned long long o = __shfl_sync(0xffffffffu, key, l);
    rank += (o > key || (o == key && l < lane)) ? 1 : 0;
  }
  const unsigned m = __ballot_sync(0xffffffffu, rank == k - 1);
  return __shfl_sync(0xffffffffu, key, __ffs(m) - 1);
}

// exclusive prefix of c over the warp; *total gets the sum
__device__ __forceinline__ int warp_excl_scan(int c, int lane, int* total) {
  int inc = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  *total = __shfl_sync(0xffffffffu, inc, 31);
  return inc - c;
}

// Rank the n <= kDartSurvCap distinct keys s[0 .. n) by counting; the entry of
// rank t < k goes to out(t, key).  EPL entries per lane.
template <int EPL, typename Key, typename Out>
__device__ __forceinline__ void dart_rank(const Key* s, int n, int k, int lane, Out out) {
  Key x[EPL];
  int r[EPL];
#pragma unroll
  for (int u = 0; u < EPL; ++u) {
    x[u] = lane + 32 * u < n ? s[lane + 32 * u] : Key(0);
    r[u] = 0;
  }
  for (int y = 0; y < n; ++y) {
    const Key o = s[y];
#pragma unroll
    for (int u = 0; u < EPL; ++u) r[u] += o > x[u] ? 1 : 0;
  }
#pragma unroll
  for (int u = 0; u < EPL; ++u)
    if (lane + 32 * u < n && r[u] < k) out(r[u], x[u]);
}

template <typename Key, typename Out>
__device__ __forceinline__ void dart_rank_any(const Key* s, int n, int k, int lane, Out out) {
  if (n <= 32) dart_rank<1>(s, n, k, lane, out);
  else if (n <= 64) dart_rank<2>(s, n, k, lane, out);
  else dart_rank<4>(s, n, k, lane, out);
}

// bf16 candidates of one tile as 32 bits: the logit's order-preserving image
// (-0 taken as +0) above 0xffff minus the element's place in the tile (< 2560)
__device__ __forceinline__ uint32_t dart_key16(uint32_t h, int loc) {
  h = h == 0x8000u ? 0u : h;
  const uint32_t o = (h & 0x8000u) ? (~h & 0xffffu) : (h | 0x8000u);
  return (o << 16) | (0xffffu - uint32_t(loc));
}

__device__ __forceinline__ DartCand dart_unkey16(uint32_t key, int tile_base) {
  const uint32_t o = key >> 16;
  const uint32_t h = (o & 0x8000u) ? (o & 0x7fffu) : (~o & 0xffffu);
  return DartCand{__uint_as_float(h << 16), tile_base + int(0xffffu - (key & 0xffffu))};
}

// the k-th largest (1 <= k <= 32) of the warp's 32 values (not NaN), equal
// values counted once per lane: a bitonic sort across the lanes, descending
__device__ __forceinline__ float warp_kth_largest_f(float v, int k, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const float o = __shfl_xor_sync(0xffffffffu, v, stride);
      const bool desc = (lane & size) == 0 || size == 32;   // this run's direction
      const bool low = (lane & stride) == 0;                  // the lower lane of the pair
      v = (low == desc) ? fmaxf(v, o) : fminf(v, o);
    }
  return __shfl_sync(0xffffffffu, v, k - 1);
}

// One warp merges a row's tile results: the combined normaliser and the top-k
// of the row's ntile * k candidates; emit(t, id, ln(p(v) + eps)) for t < k.
template <typename Emit>
__device__ __forceinline__ void dart_row_merge(const float2* part, const DartCand* cand, int ntile, int k, double c2d,
                                               double le, int row, unsigned long long* surv, int lane, Emit out) {
  const float2* pt = part + size_t(row) * ntile;
  float M = neg_inf();
  for (int t = lane; t < ntile; t += 32) M = fmaxf(M, __ldg(pt + t).x);
  M = warp_max(M);
  // sum of the partials in float64 (the terms themselves carry float32
  // rounding already: float32 2^x is as good), log2 as exponent + float32
  // log2 of the mantissa in [1, 2)
  double Z = 0.0;
  for (int t = lane; t < ntile; t += 32) {
    const float2 q = __ldg(pt + t);
    if (q.y > 0.f) Z += double(q.y) * double(exp2f(q.x - M));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, o);
  int ze;
  const double zm = frexp(Z, &ze);                          // Z = zm 2^ze, zm in [0.5, 1)
  const double lse2 = double(M) + double(ze - 1) + double(log2f(float(2.0 * zm)));
  const int nall = ntile * k;
  const int2* c = reinterpret_cast<const int2*>(cand + size_t(row) * nall);
  auto key_at = [&](int e) -> unsigned long long {
    const int2 q = __ldg(c + e);
    return q.y == kDartNone ? 0ull : dart_key(__int_as_float(q.x), q.y);
  };
  // ln(p + eps) = max(ln p, ln eps) + ln(1 + e^-|ln p - ln eps|) (le = ln eps):
  // ln p in float64, the bounded correction term in float32
  auto emit = [&](int t, unsigned long long key) {
    const DartCand x = key ? dart_unkey(key) : DartCand{neg_inf(), kDartNone};
    const double lp = x.i == kDartNone ? -INFINITY : (double(x.v) * c2d - lse2) * 0.6931471805599453;
    const double hi = lp > le ? lp : le;
    const float gap = lp > le ? float(le - lp) : float(lp - le);           // <= 0
    out(t, x.i, hi + double(log1pf(expf(gap))));
  };
  // Each tile's list is in key order, so its head is its best: the k-th best
  // of the lanes' best heads (lane l owns tiles l, l + 32, ...) comes from k
  // distinct candidates and bounds the row's k-th best from below.  Only each
  // list's prefix at or above the bound is kept.
  constexpr int kOwn = kDartMaxTiles / 32;
  unsigned long long best = 0;
#pragma unroll
  for (int u = 0; u < kOwn; ++u) {
    const int t = lane + 32 * u;
    if (t < ntile) best = max(best, key_at(t * k));
  }
  const unsigned long long thr = warp_kth_largest(best, k, lane);
  int len[kOwn];
  int cnt = 0;
#pragma unroll
  for (int u = 0; u < kOwn; ++u) {
    const int t = lane + 32 * u;
    int h = 0;
    if (t < ntile) {
      // walk the prefix four candidates at a time (independent loads)
      bool more = true;
      while (more && h < k) {
        unsigned long long x[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) x[v] = h + v < k ? key_at(t * k + h + v) : 0ull;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          if (more && x[v] != 0 && x[v] >= thr) ++h;
          else more = false;
        }
      }
    }
    len[u] = h;
    cnt += h;
  }
  int n;
  int pos = warp_excl_scan(cnt, lane, &n);
  if (n <= kDartSurvCap) {
#pragma unroll
    for (int u = 0; u < kOwn; ++u) {
      const int t = lane + 32 * u;
      for (int h = 0; h < len[u]; ++h) surv[pos++] = key_at(t * k + h);
    }
    __syncwarp();
    dart_rank_any(surv, n, k, lane, emit);
    for (int t = n + lane; t < k; t += 32) emit(t, 0ull);
    return;
  }
  // many candidates at the bound (ties): k rounds of the largest key below the last
  constexpr int kChunk = 16;
  unsigned long long prev = ~0ull;
  for (int t = 0; t < k; ++t) {
    unsigned long long b = 0;
    for (int e0 = 0; e0 < nall; e0 += 32 * kChunk) {
      unsigned long long x[kChunk];
#pragma unroll
      for (int u = 0; u < kChunk; ++u) {
        const int e = e0 + 32 * u + lane;
        x[u] = e < nall ? key_at(e) : 0ull;
      }
#pragma unroll
      for (int u = 0; u < kChunk; ++u)
        if (x[u] < prev) b = max(b, x[u]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
    if (lane == t) emit(t, b);
    prev = b;                                 // 0 once the candidates run out
  }
}

__device__ __forceinline__ __nv_bfloat162 dart_as_b2(uint32_t u) {
  __nv_bfloat162 b;
  memcpy(&b, &u, sizeof(b));
  return b;
}

template <typename Elem>
__global__ void __launch_bounds__(kDartTileWarps * 32, 3) dart_topk_tiles_kernel(DartTileArgs a) {
  using S = Slot<Elem, true>;
  constexpr int VW = S::VW;
  constexpr int NE = kDartVpt * VW;                          // elements per lane
  constexpr int MW = (NE + 31) / 32;                         // survivor-mask words
  constexpr bool kB16 = VW == 8;
  using Key = typename std::conditional<kB16, uint32_t, unsigned long long>::type;
  extern __shared__ __align__(16) unsigned char dsm[];      // per warp: the tile, in row order
  __shared__ unsigned long long s_surv[kDartTileWarps][kDartSurvCap];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long unit = long(blockIdx.x) * kDartTileWarps + warp;
  if (unit >= long(a.rows) * a.ntile) return;
  const int row = int(unit / a.ntile), tile = int(unit - long(row) * a.ntile);
  const int tile_base = tile * (32 * kDartVpt * VW);
  const Elem* x = reinterpret_cast<const Elem*>(a.logits) + size_t(row) * size_t(a.V);
  uint4* cp = reinterpret_cast<uint4*>(dsm) + warp * (kDartVpt * 32);
  S sl[kDartVpt];                                            // the lane's slots, kept packed
#pragma unroll
  for (int j = 0; j < kDartVpt; ++j) sl[j].load(x, slot_index<kDartVpt, VW>(tile, j, lane), a.V);
#pragma unroll
  for (int j = 0; j < kDartVpt; ++j) cp[j * 32 + lane] = make_uint4(sl[j].w[0], sl[j].w[1], sl[j].w[2], sl[j].w[3]);
  // the lane's largest logit (slots past the row read -inf; NaN never wins)
  float lv;
  if constexpr (kB16) {
    __nv_bfloat162 mx = __float2bfloat162_rn(neg_inf());
#pragma unroll
    for (int j = 0; j < kDartVpt; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) mx = __hmax2(mx, dart_as_b2(sl[j].w[i]));
    lv = fmaxf(__low2float(mx), __high2float(mx));
  } else {
    lv = neg_inf();
#pragma unroll
    for (int j = 0; j < kDartVpt; ++j)
#pragma unroll
      for (int e = 0; e < VW; ++e) lv = fmaxf(lv, sl[j].get(e));
  }
  // the tile's softmax partial
  const float m = warp_max(lv);
  float z = 0.f;
  if (m > neg_inf()) {
    const float2 c2 = make_float2(a.c2, a.c2), nm = make_float2(-m * a.c2, -m * a.c2);
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kDartVpt; ++j)
#pragma unroll
      for (int e = 0; e < VW; e += 2) {
        const float2 r = fma2(make_float2(sl[j].get(e), sl[j].get(e + 1)), c2, nm);
        acc = add2(acc, make_float2(ex2(r.x), ex2(r.y)));
      }
    z = acc.x + acc.y;
  }
  z = warp_sum(z);
  if (lane == 0) a.part[unit] = make_float2(m > neg_inf() ? m * a.c2 : neg_inf(), z);

  // The k-th largest of the 32 lane maxima comes from k distinct elements, so
  // the tile's top-k all have logits >= it: only those elements are kept (a
  // bit mask per lane, element q = slot * VW + e).
  const int k = a.k;
  DartCand* out = a.cand + size_t(unit) * k;
  const float tv = warp_kth_largest_f(lv, k, lane);
  uint32_t mk[MW];
#pragma unroll
  for (int w = 0; w < MW; ++w) mk[w] = 0u;
  if constexpr (kB16) {
    const __nv_bfloat162 t2 = __float2bfloat162_rn(tv);     // exact: tv is one of the logits, or -inf
#pragma unroll
    for (int j = 0; j < kDartVpt; ++j) {
      const bool ok = slot_index<kDartVpt, VW>(tile, j, lane) < a.V;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t c = ok ? __hge2_mask(dart_as_b2(sl[j].w[i]), t2) : 0u;
        const int q = j * VW + 2 * i;
        mk[q >> 5] |= ((c & 1u) | ((c >> 15) & 2u)) << (q & 31);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < kDartVpt; ++j) {
      const bool ok = slot_index<kDartVpt, VW>(tile, j, lane) < a.V;
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        const int q = j * VW + e;
        if (ok && sl[j].get(e) >= tv) mk[q >> 5] |= 1u << (q & 31);
      }
    }
  }
  int cnt = 0;
#pragma unroll
  for (int w = 0; w < MW; ++w) cnt += __popc(mk[w]);
  int n;
  int pos = warp_excl_scan(cnt, lane, &n);
  unsigned long long* surv = s_surv[warp];
  if (n <= kDartSurvCap) {
    Key* sk = reinterpret_cast<Key*>(surv);
    const Elem* te = reinterpret_cast<const Elem*>(cp);     // te[loc]: the tile's element loc
#pragma unroll
    for (int w = 0; w < MW; ++w) {
      uint32_t b = mk[w];
      while (b) {
        const int q = w * 32 + __ffs(b) - 1;
        b &= b - 1;
        const int loc = ((q / VW) * 32 + lane) * VW + (q % VW);
        if constexpr (kB16) sk[pos++] = dart_key16(reinterpret_cast<const uint16_t*>(te)[loc], loc);
        else sk[pos++] = dart_key(te[loc], tile_base + loc);
      }
    }
    __syncwarp();
    dart_rank_any(sk, n, k, lane, [&](int t, Key key) {
      if constexpr (kB16) out[t] = dart_unkey16(key, tile_base);
      else out[t] = dart_unkey(key);
    });
    for (int t = n + lane; t < k; t += 32) out[t] = DartCand{neg_inf(), kDartNone};
  } else {
    // many values tie at the bound: k rounds of the largest key below the
    // last, over the tile read again (a rare path, kept off the registers of
    // the main one)
    unsigned long long prev = ~0ull;
    for (int t = 0; t < k; ++t) {
      unsigned long long b = 0;
#pragma unroll 1
      for (int j = 0; j < kDartVpt; ++j) {
        const long base = slot_index<kDartVpt, VW>(tile, j, lane);
        if (base >= a.V) break;               // slots only grow with j
        S q;
        q.load(x, base, a.V);
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          const float v = q.get(e);
          const unsigned long long key = dart_key(v, int(base) + e);
          if (v == v && key < prev) b = max(b, key);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
      if (lane == t) out[t] = b ? dart_unkey(b) : DartCand{neg_inf(), kDartNone};
      prev = b;                               // 0 once the tile runs out
    }
  }
}

struct DartBuildArgs {
  const float2* part;                       // [R * d, ntile] tile softmax partials
  const DartCand* cand;                     // [R * d, ntile, k] tile top-k lists
  int32_t* parents;                         // [R, theta + 1]
  int32_t* tokens;                          // [R, theta + 1]
  int32_t* n_nodes;                         // [R]
  void* workspace;
  int d, k, w, theta;
  int nodes;                                // k + (d - 1) w k: T's capacity
  int ntile;
  double c2d;                               // log2(e) / T
  double ln_eps;
  double ng;                                // 0.5 ln(1 + eps)
  double pw[kDartMaxDepth];                 // 0.9^i for depth i = 1..d
  double sc[kDartMaxDepth];                 // (i + 1)^0.7
};

// T in shared memory as one array per field (a node's index is its
// generation order), so that consecutive nodes sit in consecutive banks
struct DartT {
  double* score;
  unsigned long long* s_ord;                // order-preserving image of score
  unsigned long long* k_ord;                // of the key min(score, parent key)
  int* parent;                              // node index, -1 for the root
  int* token;
  int* depth;
  int* child0;                              // first of its k children, -1 if never extended
};
constexpr int kDartNodeBytes = 3 * 8 + 4 * 4;

__device__ __forceinline__ DartT dart_t_layout(unsigned char* smem, int N) {
  DartT t;
  t.score = reinterpret_cast<double*>(smem);
  t.s_ord = reinterpret_cast<unsigned long long*>(t.score + N);
  t.k_ord = t.s_ord + N;
  t.parent = reinterpret_cast<int*>(t.k_ord + N);
  t.token = t.parent + N;
  t.depth = t.token + N;
  t.child0 = t.depth + N;
  return t;
}

// An unsigned integer with the order of the double x (x not NaN): comparisons
// then run on the integer units, not on the narrow float64 pipe.
__device__ __forceinline__ unsigned long long dart_ord(double x) {
  const unsigned long long u = static_cast<unsigned long long>(__double_as_longlong(x));
  return (u >> 63) ? ~u : (u | (1ull << 63));
}

// Selection merge in one warp over the L (<= 256) lists T[li k .. + k), each
// in (key, depth, generation) order: lane l caches the heads of lists l,
// l + 32, ...; each pick is the largest (key image, ~(depth << 16 | node)) by
// three 32-bit warp maxima, and the winning lane advances that list.
__device__ __forceinline__ void dart_select_merge(const DartT& T, int L, int k, int want, int* sel, int lane) {
  constexpr int kOwn = 8;
  unsigned long long ka[kOwn];
  unsigned kb[kOwn];
  int hd[kOwn] = {};
  auto load = [&](int v) {
    const int g = (lane + 32 * v) * k + hd[v];
    const bool live = lane + 32 * v < L && hd[v] < k;
    ka[v] = live ? T.k_ord[g] : 0ull;
    kb[v] = live ? ~static_cast<unsigned>((T.depth[g] << 16) | g) : 0u;
  };
#pragma unroll
  for (int v = 0; v < kOwn; ++v) load(v);
  unsigned long long ba = 0;
  unsigned bb = 0;
  int bv = 0;
  auto lane_best = [&]() {                         // a tree over the 8 heads
    unsigned long long ta[kOwn];
    unsigned tb[kOwn];
    int tv[kOwn];
#pragma unroll
    for (int v = 0; v < kOwn; ++v) { ta[v] = ka[v]; tb[v] = kb[v]; tv[v] = v; }
#pragma unroll
    for (int w = kOwn / 2; w >= 1; w >>= 1)
#pragma unroll
      for (int v = 0; v < w; ++v) {
        const bool hi = ta[v + w] > ta[v] || (ta[v + w] == ta[v] && tb[v + w] > tb[v]);
        ta[v] = hi ? ta[v + w] : ta[v];
        tb[v] = hi ? tb[v + w] : tb[v];
        tv[v] = hi ? tv[v + w] : tv[v];
      }
    ba = ta[0];
    bb = tb[0];
    bv = tv[0];
  };
  lane_best();
  for (int p = 0; p < want; ++p) {
    const unsigned hi = unsigned(ba >> 32), lo = unsigned(ba);
    const unsigned mh = __reduce_max_sync(0xffffffffu, hi);
    const unsigned ml = __reduce_max_sync(0xffffffffu, hi == mh ? lo : 0u);
    const bool top = hi == mh && lo == ml;
    const unsigned mb = __reduce_max_sync(0xffffffffu, top ? bb : 0u);
    if (lane == 0) sel[p] = int(~mb & 0xffffu);
    if (top && bb == mb) {                         // unique: the node index is in the key
#pragma unroll
      for (int v = 0; v < kOwn; ++v)
        if (v == bv) {
          ++hd[v];
          load(v);
        }
      lane_best();
    }
  }
  __syncwarp();
}

// Beam step in one warp: the best nn of the nact (<= 32) extension lists
// T[nb + j k .. + k), each in score order, by (score, then generation order),
// best first into act[].  A merge: lane j holds list j's head; each pick is the
// largest score image (two 32-bit warp maxima), the lowest lane on ties.
__device__ __forceinline__ void dart_beam_merge(const DartT& T, int nb, int nact, int k, int nn, int* act,
                                                int lane) {
  int h = 0, pick = -1;
  unsigned long long o = lane < nact ? T.s_ord[nb + lane * k] : 0ull;      // 0: list used up
  for (int p = 0; p < nn; ++p) {
    const unsigned hi = unsigned(o >> 32), lo = unsigned(o);
    const unsigned mh = __reduce_max_sync(0xffffffffu, hi);
    const unsigned ml = __reduce_max_sync(0xffffffffu, hi == mh ? lo : 0u);
    const unsigned win = __ballot_sync(0xffffffffu, o != 0ull && hi == mh && lo == ml);
    const int wl = __ffs(win) - 1;
    const int wh = __shfl_sync(0xffffffffu, h, wl);
    if (lane == p) pick = nb + wl * k + wh;
    if (lane == wl) {
      ++h;
      o = h < k ? T.s_ord[nb + lane * k + h] : 0ull;
    }
  }
  if (lane < nn) act[lane] = pick;
  __syncwarp();
}

constexpr int kDartRsCand = 768;          // radix select: candidates ranked at the end
constexpr int kDartRsBin = 48;            // passes go on while the bin holds more nodes

struct DartRsShared {
  unsigned long long orw[kDartBuildThreads / 32];
  int hist[256];
  unsigned long long ca[kDartRsCand];
  unsigned cb[kDartRsCand];
  int dig, above, bsize, nc;
};

// Block-wide selection of the want best of nodes [lo, lo + n) by (A[g]
// descending, then B(g) descending; B(g) = ~(depth << 16 | g), so unique),
// the node indices best first into out[]:
// 8-bit radix passes over A, from the highest bit in which the nodes differ,
// narrow the bin that holds the want-th key; the
// nodes above that bin and the bin's own nodes (at most 256) are then ranked
// by counting.  Returns false (nothing written) if a bin of more than 256
// nodes shares all of A, or want + 256 > kDartRsCand.
template <typename BKey>
__device__ __forceinline__ bool dart_radix_select(const unsigned long long* A, BKey B, int lo, int n, int want,
                                                  int* out, DartRsShared& sh, int tid) {
  if (want + 256 > kDartRsCand) return false;
  const int warp = tid >> 5, lane = tid & 31;
  unsigned long long prefix = 0, pmask = 0;
  int need = want, bsize = n;
  int shift = 56;
  if (n > 256) {                                        // bits above the highest differing one are common
    const unsigned long long ref = A[lo];
    unsigned long long x = 0;
    for (int g = lo + tid; g < lo + n; g += kDartBuildThreads) x |= A[g] ^ ref;
    const unsigned xh = __reduce_or_sync(0xffffffffu, unsigned(x >> 32));
    const unsigned xl = __reduce_or_sync(0xffffffffu, unsigned(x));
    if (lane == 0) sh.orw[warp] = (static_cast<unsigned long long>(xh) << 32) | xl;
    __syncthreads();
    x = 0;
#pragma unroll
    for (int v = 0; v < kDartBuildThreads / 32; ++v) x |= sh.orw[v];
    if (x == 0) return false;                           // more than 256 nodes share A
    shift = 63 - __clzll(static_cast<long long>(x)) - 7;                // digit = the 8 bits below it
  }
  for (; shift > -8 && bsize > kDartRsBin; shift -= 8) {
    const unsigned long long dmask = shift >= 0 ? 255ull << shift : 255ull >> -shift;
    sh.hist[tid] = 0;                                   // 256 threads, 256 bins
    __syncthreads();
    for (int g = lo + tid; g < lo + n; g += kDartBuildThreads) {
      const unsigned long long a = A[g];
      if ((a & pmask) == prefix)
        atomicAdd(&sh.hist[shift >= 0 ? (a >> shift) & 255u : (a << -shift) & 255u], 1);
    }
    __syncthreads();
    if (warp == 0) {                                    // lane l: bins 255 - 8l .. 248 - 8l
      int c[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) { c[j] = sh.hist[255 - 8 * lane - j]; tot += c[j]; }
      int dummy;
      int run = warp_excl_scan(tot, lane, &dummy);
      int found = -1, above = 0, bs = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (found < 0 && run < need && run + c[j] >= need) { found = 255 - 8 * lane - j; above = run; bs = c[j]; }
        run += c[j];
      }
      const unsigned m = __ballot_sync(0xffffffffu, found >= 0);
      if (lane == __ffs(m) - 1) { sh.dig = found; sh.above = above; sh.bsize = bs; }
    }
    __syncthreads();
    need -= sh.above;
    bsize = sh.bsize;
    const unsigned long long dg = static_cast<unsigned long long>(sh.dig);
    prefix |= shift >= 0 ? dg << shift : dg >> -shift;
    pmask |= dmask;
  }
  if (bsize > 256) return false;
  // gather the nodes above the bin (want - need of them) and the bin's nodes
  if (tid == 0) sh.nc = 0;
  __syncthreads();
  for (int g = lo + tid; g < lo + n; g += kDartBuildThreads) {
    const unsigned long long a = A[g];
    if ((a & pmask) >= prefix) {
      const int at = atomicAdd(&sh.nc, 1);
      sh.ca[at] = a;
      sh.cb[at] = B(g);
    }
  }
  __syncthreads();
  const int nc = sh.nc;
  for (int x = tid; x < nc; x += kDartBuildThreads) {
    const unsigned long long xa = sh.ca[x];
    const unsigned xb = sh.cb[x];
    int rk = 0;
    for (int y = 0; y < nc; ++y) rk += (sh.ca[y] > xa || (sh.ca[y] == xa && sh.cb[y] > xb)) ? 1 : 0;
    if (rk < want) out[rk] = int(~xb & 0xffffu);
  }
  __syncthreads();
  return true;
}

__global__ void __launch_bounds__(kDartBuildThreads) dart_build_kernel(DartBuildArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const DartT T = dart_t_layout(smem, a.nodes);                    // [k + (d - 1) w k]
  __shared__ int s_tok[kDartMaxDepth][kDartMaxK];
  __shared__ double s_inc[kDartMaxDepth][kDartMaxK];
  __shared__ int s_active[kDartMaxW];
  __shared__ int s_sel[kDartMaxTheta];
  // the depth-first layout's subtree sizes, parents' selection indices and rows
  // (first the row merges' survivors, 8 warps x kDartSurvCap keys)
  __shared__ __align__(16) int s_work[3 * (kDartMaxTheta + 1)];
  static_assert(sizeof(s_work) >= kDartBuildThreads / 32 * kDartSurvCap * 8, "merge scratch");

  DartRsShared& rs = *reinterpret_cast<DartRsShared*>(s_work);                  // by phase
  static_assert(sizeof(s_work) >= sizeof(DartRsShared), "radix select scratch");
  const int r = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d = a.d, k = a.k, w = a.w;
  // the selection's second sort key: smaller depth, then older
  auto bkey = [&](int g) { return ~static_cast<unsigned>((T.depth[g] << 16) | g); };
  if (r == 0 && tid == 0) *reinterpret_cast<int*>(a.workspace) = 0;

  // ---- per offset i (one warp each): the row's top-k from its tile lists and
  // eq. (10)'s increment of each pick at depth i + 1, computed once:
  // (0.9^(i+1) ln(p(v) + eps) + 0.5 ln(1 + eps)) / (i + 2)^0.7
  unsigned long long* s_mrg = reinterpret_cast<unsigned long long*>(s_work) + warp * kDartSurvCap;
  for (int i = warp; i < d; i += kDartBuildThreads / 32)
    dart_row_merge(a.part, a.cand, a.ntile, k, a.c2d, a.ln_eps, r * d + i, s_mrg, lane, [&](int t, int id, double lpv) {
      s_tok[i][t] = id;
      s_inc[i][t] = (a.pw[i] * lpv + a.ng) / a.sc[i];
    });
  __syncthreads();

  // ---- beam over depths.  T[0 .. k) are the root's children; at depth i >= 2
  // active path j's k extensions are T[nb + j k .. + k) (all threads build
  // them); warp 0 then keeps the w best as the next active paths, in order.
  for (int t = tid; t < k; t += kDartBuildThreads) {
    const double sv = s_inc[0][t];
    T.score[t] = sv;
    T.s_ord[t] = T.k_ord[t] = dart_ord(sv);
    T.parent[t] = -1;
    T.token[t] = s_tok[0][t];
    T.depth[t] = 1;
    T.child0[t] = -1;
  }
  int nact = min(w, k);
  int base = 0, count = k;
  // depth 1: the root's list, in score order (the picks come in logit order)
  for (int j = tid; j < nact; j += kDartBuildThreads) s_active[j] = j;
  __syncthreads();
  for (int i = 2; i <= d; ++i) {
    const int nb = base + count;
    for (int q = tid; q < nact * k; q += kDartBuildThreads) {
      const int j = q / k, t = q - j * k;
      const int par = s_active[j], g = nb + q;
      const double sc = T.score[par] + s_inc[i - 1][t];
      const unsigned long long so = dart_ord(sc), pk = T.k_ord[par];
      T.score[g] = sc;
      T.s_ord[g] = so;
      T.k_ord[g] = so < pk ? so : pk;                              // key = min(score, parent key)
      T.parent[g] = par;
      T.token[g] = s_tok[i - 1][t];
      T.depth[g] = i;
      T.child0[g] = -1;
    }
    __syncthreads();
    for (int j = tid; j < nact; j += kDartBuildThreads) T.child0[s_active[j]] = nb + j * k;
    const int cnt = nact * k, nnext = min(w, cnt);
    if (i < d && warp == 0) dart_beam_merge(T, nb, nact, k, nnext, s_active, lane);
    __syncthreads();
    base = nb;
    count = cnt;
    nact = nnext;
  }
  const int total = base + count;
  const int want = min(a.theta, total);

  // ---- selection: the want best nodes of T by (key, then smaller depth, then
  // generation order), best first.  Keys never increase along a path and ties
  // go to the shallower node, so this set is ancestor-closed.  T is a run of
  // lists of k nodes (the root's, then each extended path's extensions), each
  // already in this order, so the selection is a merge of all of them.
  if (!dart_radix_select(T.k_ord, bkey, 0, total, want, s_sel, rs, tid) && warp == 0)
    dart_select_merge(T, total / k, k, want, s_sel, lane);
  __syncthreads();

  // ---- the tree, depth first from the root, children in selection order:
  // subtree sizes bottom-up, then each node's row = its parent's row + 1 +
  // the sizes of its earlier-selected siblings, top-down.  T.child0 now holds
  // the node's selection index.
  int* s_sub = s_work;
  int* s_pq = s_sub + (kDartMaxTheta + 1);
  int* s_row = s_pq + (kDartMaxTheta + 1);
  for (int q = tid; q < want; q += kDartBuildThreads) T.child0[s_sel[q]] = q;
  __syncthreads();
  for (int q = tid; q < want; q += kDartBuildThreads) {
    const int pa = T.parent[s_sel[q]];
    s_pq[q] = pa < 0 ? -1 : T.child0[pa];
    s_sub[q] = 1;
  }
  __syncthreads();
  for (int lev = d; lev >= 2; --lev) {
    for (int q = tid; q < want; q += kDartBuildThreads)
      if (T.depth[s_sel[q]] == lev) atomicAdd(&s_sub[s_pq[q]], s_sub[q]);
    __syncthreads();
  }
  // offset of each node below its parent's row: 1 + the sizes of the siblings
  // selected before it
  for (int q = tid; q < want; q += kDartBuildThreads) {
    const int pq = s_pq[q];
    int before = 1;
    for (int y = 0; y < q; ++y) before += s_pq[y] == pq ? s_sub[y] : 0;
    s_row[q] = before;
  }
  __syncthreads();
  for (int lev = 2; lev <= d; ++lev) {           // depth-1 rows are their offsets (root row 0)
    for (int q = tid; q < want; q += kDartBuildThreads)
      if (T.depth[s_sel[q]] == lev) s_row[q] += s_row[s_pq[q]];
    __syncthreads();
  }
  int32_t* par_out = a.parents + size_t(r) * (a.theta + 1);
  int32_t* tok_out = a.tokens + size_t(r) * (a.theta + 1);
  for (int q = tid; q <= a.theta; q += kDartBuildThreads) {
    if (q == 0 || q > want) { par_out[q] = -1; tok_out[q] = 0; }
  }
  for (int q = tid; q < want; q += kDartBuildThreads) {
    const int pq = s_pq[q];
    par_out[s_row[q]] = pq < 0 ? 0 : s_row[pq];
    tok_out[s_row[q]] = T.token[s_sel[q]];
  }
  if (tid == 0) a.n_nodes[r] = want + 1;
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
  if (ntile > kDartMaxTiles) return false;
  p->ntile = int(ntile);
  const size_t rows = size_t(R) * d;
  size_t off = kHeaderBytes;
  p->part_off = off;
  off = align256(off + rows * ntile * sizeof(float2));
  p->cand_off = off;
  off = align256(off + rows * ntile * k * sizeof(DartCand));
  p->total = off;
  const size_t nodes = size_t(k) + size_t(d - 1) * w * k;
  p->build_smem = nodes * kDartNodeBytes;            // T; the rest is static
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
  const size_t tsmem = size_t(kDartTileWarps) * kDartVpt * 32 * 16;       // each warp's tile
  if (cudaFuncSetAttribute(tfn, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
    return SPECV_ERR_CUDA;                                                  // three 48 KB CTAs per SM
  if (cudaLaunchKernel(tfn, dim3(unsigned((units + kDartTileWarps - 1) / kDartTileWarps)), dim3(kDartTileWarps * 32),
                       targs, tsmem, st) != cudaSuccess)
    return SPECV_ERR_CUDA;
  DartBuildArgs ba;
  ba.part = ta.part;
  ba.cand = ta.cand;
  ba.ntile = p.ntile;
  ba.c2d = double(ta.c2);
  ba.ln_eps = log(kDartEps);
  ba.parents = parents;
  ba.tokens = tokens;
  ba.n_nodes = n_nodes;
  ba.workspace = workspace;
  ba.d = d;
  ba.k = k;
  ba.w = w;
  ba.theta = theta;
  ba.nodes = int(size_t(k) + size_t(d - 1) * w * k);
  // eq. (10)'s constants, from the host's libm (the float64 pipe is narrow)
  ba.ng = 0.5 * log(1.0 + kDartEps);
  for (int i = 1; i <= kDartMaxDepth; ++i) {
    ba.pw[i - 1] = pow(0.9, double(i));
    ba.sc[i - 1] = pow(double(i + 1), 0.7);
  }
  if (cudaFuncSetAttribute(reinterpret_cast<const void*>(&dart_build_kernel), cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(p.build_smem)) != cudaSuccess)
    return SPECV_ERR_CUDA;
  void* bargs[] = {&ba};
  if (cudaLaunchKernel(reinterpret_cast<const void*>(&dart_build_kernel), dim3(unsigned(R)), dim3(kDartBuildThreads),
                       bargs, p.build_smem, st) != cudaSuccess)
    return SPECV_ERR_CUDA;
  return SPECV_OK;
}
