// The DSpark Markov draft head (sm_103a).
//
// Method (DSpark paper guide, Markov head): p_k(v | x_0, x_<k) =
// softmax(U_k(v) + B(x_{k-1}, v)) with the low-rank factorisation B = W1 W2
// (W1 [V, r] used as a row lookup, W2 [r, V] as a logit projection), sampled
// position by position from the anchor x_0.
//
// Per step k (x_{k-1} -> x_k), tensor-core form (rank a multiple of 64, at most
// 256; V a multiple of 8; 16-byte aligned tensors):
//   markov_tc       persistent: one CTA per SM, each owning 256 requests (two
//                   M = 128 blocks) and a strided set of 64-column vocabulary
//                   tiles.  The W1[x_{k-1}] rows are gathered once into shared
//                   memory (K-major, 128-byte swizzle); a TMA warp streams
//                   [rank x 64] tiles of W2 (read in place as an MN-major
//                   operand) through a two-stage ring; one thread issues tcgen05.mma
//                   (M = 128, N = 64, K = 16, bf16 -> float32) into a
//                   double-buffered TMEM accumulator; eight epilogue warps read
//                   TMEM, add U_k, write L and the tile's softmax partials.
// CUDA-core form (any other shape):
//   markov_logits   L = U_k + W1[x_{k-1}] . W2 for a [BM x BN] output tile,
//                   float32 accumulation; the epilogue writes L (float32 or
//                   bf16) and the tile's softmax partials (max * c2,
//                   sum 2^(L*c2 - max*c2)) or, at T = 0, (max, argmax).
//   markov_sample   one warp per request: combines the tile partials, picks the
//                   tile holding u * Z and rescans its BN logits (inverse CDF
//                   over ascending ids), or takes the argmax at T = 0.
#include <atomic>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "host_common.h"
#include "tc.cuh"

namespace specv {

constexpr int kMkBM = 32;        // requests per tile
constexpr int kMkBN = 128;       // vocabulary columns per tile
constexpr int kMkBK = 64;        // rank chunk
constexpr int kMkThreads = 256;  // 8 warps x 4 rows, 32 lanes x 4 columns

struct MarkovPart {
  float a;   // T > 0: tile max * c2;  T = 0: tile max
  float b;   // T > 0: sum 2^(L*c2 - a);  T = 0: argmax index (as int bits)
};

struct MarkovArgs {
  const uint16_t* U;          // [R, gamma, V] bf16
  const uint16_t* W1;         // [V, rank] bf16
  const uint16_t* W2;         // [rank, V] bf16
  const int32_t* anchor;      // [R]
  const float* uniforms;      // [R, gamma]
  int32_t* tokens;            // [R, gamma]
  void* logits;               // output logits base: [R, lstride_r] rows of V (f32 or bf16); null: none kept
                              // (tensor-core form only: the sampler recomputes its tile)
  int logits_bf16;
  long lstride_r;             // elements between consecutive requests in `logits`
  long step_off;              // element offset of this step's row inside a request
  MarkovPart* part;           // [R, ntile]
  void* workspace;
  int R, gamma, V, rank, k;   // k = 1 .. gamma
  int ntile;
  float c2;                   // log2(e)/T, 0 at T = 0
  int greedy;
  int tile_w;                 // vocabulary columns per partial (64 or 128)
};

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// two floats rounded to bf16 (round to nearest even) and packed, x in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float round_to_bf16(float x) {
  // round-to-nearest-even to bf16, back to float (finite inputs)
  uint32_t u = __float_as_uint(x);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return __uint_as_float(u & 0xFFFF0000u);
}

// float(bf16 low half of w) + lo and float(bf16 high half) + hi, each one f32
// add rounded to nearest (the conversions are exact)
__device__ __forceinline__ float2 add_bf16x2(uint32_t w, float lo, float hi) {
  float x, y;
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n add.rn.f32.bf16 %0, l, %3;\n add.rn.f32.bf16 %1, h, %4;\n}"
      : "=f"(x), "=f"(y) : "r"(w), "f"(lo), "f"(hi));
  return make_float2(x, y);
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// One row's 64-column chunk of L = U + W1[x] . W2: u holds its 64 bf16 U
// values as eight 16-byte granules, acc0 / acc1 its accumulator columns 0-31 /
// 32-63; rounded to bf16 when that is the draw precision.
__device__ __forceinline__ void chunk_logits(const uint4 (&u)[8], const float (&acc0)[32], const float (&acc1)[32],
                                             bool to_bf16, float (&L)[64]) {
#pragma unroll
  for (int cc = 0; cc < 8; ++cc) {
    const uint32_t wv[4] = {u[cc].x, u[cc].y, u[cc].z, u[cc].w};
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const int j = 8 * cc + e;
      float2 x = j < 32 ? add_bf16x2(wv[e >> 1], acc0[j], acc0[j + 1]) : add_bf16x2(wv[e >> 1], acc1[j - 32], acc1[j - 31]);
      if (to_bf16) {
        const uint32_t pk = pack_bf16x2(x.x, x.y);
        x = make_float2(__uint_as_float(pk << 16), __uint_as_float(pk & 0xFFFF0000u));
      }
      L[j] = x.x;
      L[j + 1] = x.y;
    }
  }
}

// The tile partial of one row's 64-column chunk whose columns past V hold -inf:
// (max, argmax) at T = 0, else (max * c2, sum 2^(L * c2 - max * c2)).  Maxima
// by three-input max in a depth-4 tree; the sum in four packed chains.
__device__ __forceinline__ MarkovPart chunk_partial(const float (&L)[64], int n0, const MarkovArgs& a) {
  MarkovPart p;
  if (a.greedy) {
    float m = L[0];
    int idx = n0;
#pragma unroll
    for (int j = 1; j < 64; ++j)
      if (L[j] > m) { m = L[j]; idx = n0 + j; }
    p.a = m;
    p.b = __int_as_float(idx);
    return p;
  }
  float m1[22], m2[8];
#pragma unroll
  for (int j = 0; j < 21; ++j) m1[j] = max3(L[3 * j], L[3 * j + 1], L[3 * j + 2]);
  m1[21] = L[63];
#pragma unroll
  for (int j = 0; j < 7; ++j) m2[j] = max3(m1[3 * j], m1[3 * j + 1], m1[3 * j + 2]);
  m2[7] = m1[21];
  const float mx = max3(max3(m2[0], m2[1], m2[2]), max3(m2[3], m2[4], m2[5]), fmaxf(m2[6], m2[7]));
  const float m_c2 = mx * a.c2;
  const float2 c2v = make_float2(a.c2, a.c2), mv = make_float2(-m_c2, -m_c2);
  float2 z[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
  for (int j = 0; j < 64; j += 2) {
    const float2 tt = fma2(make_float2(L[j], L[j + 1]), c2v, mv);
    z[(j >> 1) & 3] = add2(z[(j >> 1) & 3], make_float2(ex2(tt.x), ex2(tt.y)));
  }
  p.a = m_c2;
  p.b = ((z[0].x + z[0].y) + (z[1].x + z[1].y)) + ((z[2].x + z[2].y) + (z[3].x + z[3].y));
  return p;
}

// A tile partial, stored with an L2 eviction policy: evict_last keeps the
// partials (R * ceil(V / 64) * 8 bytes) resident through the step's streamed
// U and logit traffic until the sampler reads them.
__device__ __forceinline__ void store_part(MarkovPart* dst, MarkovPart v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;" ::"l"(dst), "f"(v.a), "f"(v.b), "l"(policy)
               : "memory");
}

__device__ __forceinline__ int prev_token(const MarkovArgs& a, int r) {
  return a.k == 1 ? a.anchor[r] : a.tokens[size_t(r) * a.gamma + (a.k - 2)];
}

__global__ void __launch_bounds__(kMkThreads) markov_logits_kernel(MarkovArgs a) {
  __shared__ float s_w1[kMkBM][kMkBK + 1];
  __shared__ __align__(16) float s_w2[kMkBK][kMkBN];
  __shared__ int s_prev[kMkBM];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int v0 = blockIdx.x * kMkBN;
  const int r0 = blockIdx.y * kMkBM;
  if (a.k == 1 && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *reinterpret_cast<int*>(a.workspace) = 0;
  if (threadIdx.x < kMkBM) {
    const int r = r0 + threadIdx.x;
    int x = -1;
    if (r < a.R) {
      x = prev_token(a, r);
      if (x < 0 || x >= a.V) x = -1;
    }
    s_prev[threadIdx.x] = x;
  }
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[i][c] = 0.f;
  __syncthreads();
  for (int kb = 0; kb < a.rank; kb += kMkBK) {
    for (int e = threadIdx.x; e < kMkBM * kMkBK; e += kMkThreads) {
      const int i = e / kMkBK, j = e % kMkBK;
      const int x = s_prev[i];
      s_w1[i][j] = (x >= 0 && kb + j < a.rank) ? bf16_to_f32(a.W1[size_t(x) * a.rank + kb + j]) : 0.f;
    }
    for (int e = threadIdx.x; e < kMkBK * kMkBN; e += kMkThreads) {
      const int j = e / kMkBN, c = e % kMkBN;
      const int v = v0 + c;
      s_w2[j][c] = (kb + j < a.rank && v < a.V) ? bf16_to_f32(a.W2[size_t(kb + j) * a.V + v]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int j = 0; j < kMkBK; ++j) {
      const float4 b = *reinterpret_cast<const float4*>(&s_w2[j][lane * 4]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float w = s_w1[warp * 4 + i][j];
        acc[i][0] = fmaf(w, b.x, acc[i][0]);
        acc[i][1] = fmaf(w, b.y, acc[i][1]);
        acc[i][2] = fmaf(w, b.z, acc[i][2]);
        acc[i][3] = fmaf(w, b.w, acc[i][3]);
      }
    }
    __syncthreads();
  }
  // epilogue: L = U + bias, store, tile partials
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + warp * 4 + i;
    if (r >= a.R) continue;                       // warp-uniform
    float L[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int v = v0 + lane * 4 + c;
      if (v < a.V) {
        float x = bf16_to_f32(a.U[(size_t(r) * a.gamma + (a.k - 1)) * a.V + v]) + acc[i][c];
        if (a.logits_bf16) x = round_to_bf16(x);
        L[c] = x;
      } else {
        L[c] = neg_inf();
      }
    }
    const size_t base = size_t(r) * a.lstride_r + a.step_off;
    if (a.logits) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int v = v0 + lane * 4 + c;
        if (v < a.V) {
          if (a.logits_bf16) reinterpret_cast<uint16_t*>(a.logits)[base + v] = uint16_t(__float_as_uint(L[c]) >> 16);
          else reinterpret_cast<float*>(a.logits)[base + v] = L[c];
        }
      }
    }
    MarkovPart mp;
    if (a.greedy) {
      float m = L[0];
      int idx = v0 + lane * 4;
#pragma unroll
      for (int c = 1; c < 4; ++c)
        if (L[c] > m) { m = L[c]; idx = v0 + lane * 4 + c; }
      warp_argmax(m, idx);
      mp.a = m;
      mp.b = __int_as_float(idx);
    } else {
      float m = fmaxf(fmaxf(L[0], L[1]), fmaxf(L[2], L[3]));
      m = warp_max(m);
      const float m_c2 = m * a.c2;
      float z = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) z += ex2(fmaf(L[c], a.c2, -m_c2));
      z = warp_sum(z);
      mp.a = m_c2;
      mp.b = z;
    }
    if (lane == 0) a.part[size_t(r) * a.ntile + blockIdx.x] = mp;
  }
}

// One CTA per request: combine the tile partials, pick the tile holding u * Z
// (prefix over tiles in index order), rescan its logits; T = 0 takes the argmax.
constexpr int kSampleThreads = 256;
constexpr int kSampleWarps = kSampleThreads / 32;
constexpr int kSampleMaxPer = 16;     // tiles per thread: at most 4096 tiles per row
constexpr int kSampleMaxRank = 256;   // rank of the tensor-core form, whose tiles may be recomputed

__global__ void __launch_bounds__(kSampleThreads, 4) markov_sample_kernel(MarkovArgs a) {
  __shared__ float s_e[kSampleMaxRank];  // W1[x_{k-1}] when the tile is recomputed
  __shared__ float s_wsum[kSampleWarps][64];   // per-warp rank sums of the recomputed tile
  __shared__ float s_chunk[1][64];       // the recomputed tile
  __shared__ float s_f[kSampleWarps];
  __shared__ int s_i[kSampleWarps];
  __shared__ int s_sel;
  __shared__ float s_base, s_target;
  __shared__ MarkovPart s_part[kSampleMaxPer * kSampleThreads * 9 / 8];   // tile t at t + t / 8
  pdl_wait_primary();                      // the logits and partials of this step are complete
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x;
  const MarkovPart* part = a.part + size_t(r) * a.ntile;
  // T > 0: the row's tile partials go through shared memory, loaded first (they
  // do not wait on the previous token) and coalesced: thread i takes tiles
  // i, i + 256, ...; each thread later reads back its contiguous run, which the
  // one 8-byte pad per 8 tiles keeps free of bank conflicts.
  if (!a.greedy) {
#pragma unroll
    for (int j = 0; j < kSampleMaxPer; ++j) {
      const int t = j * kSampleThreads + threadIdx.x;
      if (t < a.ntile) s_part[t + (t >> 3)] = part[t];
    }
  }
  const int x_prev = prev_token(a, r);
  const float u = a.greedy ? 0.f : a.uniforms[size_t(r) * a.gamma + (a.k - 1)];
  const bool bad_in = x_prev < 0 || x_prev >= a.V || (!a.greedy && !(u >= 0.f && u < 1.f));
  // the conditioning row W1[x_{k-1}] of a tile recompute, fetched while the
  // partials are combined (it does not depend on the selected tile)
  if (a.logits == nullptr && !a.greedy && !bad_in)
    for (int j = threadIdx.x; j < a.rank; j += kSampleThreads) s_e[j] = bf16_to_f32(a.W1[size_t(x_prev) * a.rank + j]);
  int tok = -1;
  if (a.greedy) {
    float v = neg_inf();
    int i = 0x7fffffff;
    for (int t = threadIdx.x; t < a.ntile; t += kSampleThreads) {
      const MarkovPart p = part[t];
      const int pi = __float_as_int(p.b);
      if (p.a > v || (p.a == v && pi < i)) { v = p.a; i = pi; }
    }
    warp_argmax(v, i);
    if (lane == 0) { s_f[warp] = v; s_i[warp] = i; }
    __syncthreads();
    if (warp == 0) {
      v = lane < kSampleWarps ? s_f[lane] : neg_inf();
      i = lane < kSampleWarps ? s_i[lane] : 0x7fffffff;
      warp_argmax(v, i);
      if (lane == 0) {
        a.tokens[size_t(r) * a.gamma + (a.k - 1)] = bad_in ? -1 : i;
        if (bad_in) record_device_error(a.workspace, SPECV_ERR_DEVICE_DATA);
      }
      pdl_launch_dependents();
    }
    return;
  }
  // this thread's contiguous run of tiles, cached in registers; row maximum of
  // the tile maxima (already times c2)
  __syncthreads();
  const int per = (a.ntile + kSampleThreads - 1) / kSampleThreads;     // <= kSampleMaxPer
  const int t0 = threadIdx.x * per, t1 = min(a.ntile, t0 + per);
  float pa[kSampleMaxPer], pb[kSampleMaxPer];
  float M = neg_inf();
#pragma unroll
  for (int j = 0; j < kSampleMaxPer; ++j) {
    pa[j] = neg_inf();
    pb[j] = 0.f;
    if (t0 + j < t1) {
      const int t = t0 + j;
      const MarkovPart p = s_part[t + (t >> 3)];
      pa[j] = p.a;
      pb[j] = p.b;
      M = fmaxf(M, p.a);
    }
  }
  M = warp_max(M);
  if (lane == 0) s_f[warp] = M;
  __syncthreads();
  M = neg_inf();
#pragma unroll
  for (int w = 0; w < kSampleWarps; ++w) M = fmaxf(M, s_f[w]);
  __syncthreads();                                 // s_f is reused below
  // block-wide inclusive scan of the tile masses
  float lsum = 0.f;
#pragma unroll
  for (int j = 0; j < kSampleMaxPer; ++j) {
    pb[j] = pb[j] > 0.f ? pb[j] * ex2(pa[j] - M) : 0.f;     // tile mass relative to the row maximum
    lsum += pb[j];
  }
  float incl = warp_inclusive_scan(lsum);
  if (lane == 31) s_f[warp] = incl;
  __syncthreads();
  float wpre = 0.f, total = 0.f;
#pragma unroll
  for (int w = 0; w < kSampleWarps; ++w) {
    const float x = s_f[w];
    if (w < warp) wpre += x;
    total += x;
  }
  incl += wpre;
  const float target = u * total;
  if (threadIdx.x == 0) {
    s_sel = -1;
    s_target = target;
  }
  __syncthreads();
  // first thread whose run passes the target; it walks its run (rounding may
  // leave none: then the last thread with mass takes its last tile with mass)
  const bool hit = incl > target && t1 > t0 && lsum > 0.f;
  const unsigned wb = __ballot_sync(0xffffffffu, hit);
  if (lane == 0) s_i[warp] = wb ? warp * 32 + __ffs(wb) - 1 : 0x7fffffff;
  __syncthreads();
  int first = 0x7fffffff;
#pragma unroll
  for (int w = 0; w < kSampleWarps; ++w) first = min(first, s_i[w]);
  if (first == 0x7fffffff) {                      // block-uniform
    __syncthreads();                               // every thread has read s_i
    const unsigned mb = __ballot_sync(0xffffffffu, lsum > 0.f);
    if (lane == 0) s_i[warp] = mb ? warp * 32 + 31 - __clz(mb) : -1;
    __syncthreads();
    int last = -1;
#pragma unroll
    for (int w = 0; w < kSampleWarps; ++w) last = max(last, s_i[w]);
    first = last;
  }
  if (int(threadIdx.x) == first) {
    float run = incl - lsum;
    int sel = -1;
    float base = 0.f;
    bool done = false;
#pragma unroll
    for (int j = 0; j < kSampleMaxPer; ++j) {
      const float m = pb[j];
      if (!done && m > 0.f) {
        sel = t0 + j;
        base = run;
        done = run + m > target;
      }
      if (!done) run += m;
    }
    s_sel = sel;
    s_base = base;
  }
  __syncthreads();
  const int sel = s_sel;
  bool bad = bad_in || sel < 0;
  if (a.logits == nullptr) {
    // No logits were kept (tensor-core form, tile_w = 64): recompute the
    // selected tile's 64 logits, L(v) = U_k(v) + sum_j W1[x_{k-1}, j] W2[j, v].
    // Warp w takes rank rows 32w .. 32w + 31 and lane l columns 2l, 2l + 1: one
    // 4-byte load per row, all independent, sixteen issued at a time (eight and
    // all thirty-two were measured slower); the warps' float32 sums are then
    // added in warp order.
    // Warp w takes rank rows 32w .. 32w + 31 and lane l columns 2l, 2l + 1: one
    // 4-byte load per row, all independent, sixteen issued at a time (eight and
    // all thirty-two were measured slower); the warps' float32 sums are then
    // added in warp order.
    const int v2 = sel * 64 + 2 * lane;                  // this lane's column pair (s_e was filled at the start)
    const int per_w = (a.rank + kSampleWarps - 1) / kSampleWarps;
    float2 acc = make_float2(0.f, 0.f);
    if (!bad && v2 < a.V) {
      const int j0 = warp * per_w, j1 = min(a.rank, j0 + per_w);
      const uint16_t* w2 = a.W2 + v2;
#pragma unroll 16
      for (int j = j0; j < j1; ++j) {
        const uint32_t pr = *reinterpret_cast<const uint32_t*>(w2 + size_t(j) * a.V);   // V even: 4-byte aligned
        acc = fma2(make_float2(s_e[j], s_e[j]), make_float2(__uint_as_float(pr << 16), __uint_as_float(pr & 0xFFFF0000u)),
                   acc);
      }
    }
    s_wsum[warp][2 * lane] = acc.x;
    s_wsum[warp][2 * lane + 1] = acc.y;
    __syncthreads();
    if (threadIdx.x < 64) {
      const int c = threadIdx.x, v = sel * 64 + c;
      float x = neg_inf();
      if (!bad && v < a.V) {
        float dot = 0.f;
#pragma unroll
        for (int w = 0; w < kSampleWarps; ++w) dot += s_wsum[w][c];
        x = bf16_to_f32(a.U[(size_t(r) * a.gamma + (a.k - 1)) * a.V + v]) + dot;
        if (a.logits_bf16) x = __uint_as_float(pack_bf16x2(x, 0.f) << 16);
      }
      s_chunk[0][c] = x;                       // the tile's logits, in column order
    }
    __syncthreads();
  }
  if (warp != 0) return;                   // warp 0 triggers the next step once the token is written
  if (!bad) {
    // rescan the selected tile's columns in index order
    const MarkovPart p = part[sel];
    const float sc = ex2(p.a - M);
    const size_t rowbase = size_t(r) * a.lstride_r + a.step_off;
    const int cpl = a.tile_w / 32;             // columns per lane: 2 or 4
    float w[4];
    float ls = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int v = sel * a.tile_w + lane * cpl + c;
      float x = neg_inf();
      if (c < cpl && v < a.V) {
        if (a.logits == nullptr) x = s_chunk[0][lane * cpl + c];
        else x = a.logits_bf16 ? bf16_to_f32(reinterpret_cast<const uint16_t*>(a.logits)[rowbase + v])
                               : reinterpret_cast<const float*>(a.logits)[rowbase + v];
      }
      w[c] = __fmul_rn(ex2(fmaf(x, a.c2, -p.a)), sc);
      ls += w[c];
    }
    const float inc = warp_inclusive_scan(ls);
    float accv = s_base + (inc - ls);
    int cand = 0x7fffffff, last = -1;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (c >= cpl) break;
      accv += w[c];
      const int v = sel * a.tile_w + lane * cpl + c;
      if (w[c] > 0.f) last = v;
      if (cand == 0x7fffffff && accv > s_target && w[c] > 0.f) cand = v;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
      last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
    }
    tok = cand != 0x7fffffff ? cand : last;
    if (tok < 0) bad = true;
  }
  if (lane == 0) {
    a.tokens[size_t(r) * a.gamma + (a.k - 1)] = bad ? -1 : tok;
    if (bad) record_device_error(a.workspace, SPECV_ERR_DEVICE_DATA);
  }
  pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// tensor-core form
constexpr int kTcBN = 64;                 // vocabulary columns per tile (UMMA N)
constexpr int kTcBM = 128;                // requests per CTA (UMMA M)
constexpr int kTcMaxKC = 4;               // 64-wide rank chunks (rank <= 256)
constexpr int kTcEpiWarps = 8;            // two groups of four: group g takes the tiles i with i % 2 == g
constexpr int kTcThreads = (kTcEpiWarps + 2) * 32;   // + TMA warp + MMA warp
constexpr uint32_t kTcTmemCols = 128;     // two accumulator buffers of 64 columns
constexpr uint32_t kTcRowBytes = 128;     // one swizzled row
constexpr size_t kTcSmemE = size_t(kTcMaxKC) * kTcBM * kTcRowBytes;        // 64 KB: W1 rows
constexpr size_t kTcStageB = size_t(kTcMaxKC) * 64 * kTcRowBytes;          // 32 KB: one W2 tile [rank][64]
constexpr size_t kTcStageU = size_t(kTcBM) * kTcRowBytes;                   // 16 KB: one U tile
constexpr size_t kTcSmemL = size_t(kTcEpiWarps) * 2 * 32 * kTcRowBytes;    // 64 KB: logit staging per warp
// NS stages of the W2 and U rings: two when logits are stored (the staging
// takes the rest of shared memory), three when they are not
__host__ __device__ constexpr size_t tc_smem(int ns, bool store) {
  return kTcSmemE + size_t(ns) * (kTcStageB + kTcStageU) + (store ? kTcSmemL : 0) + 1024;
}
constexpr uint32_t kTcMaxPolls = 1u << 22;   // bound on every mbarrier wait
constexpr uint32_t kTcIdesc = tc::idesc_bf16_f32(kTcBM, kTcBN, true);   // B = W2, MN-major

struct MarkovTcArgs {
  MarkovArgs m;
  int nkc;          // rank / 64
  int ntiles;       // ceil(V / 64)
  int per_mb;       // CTAs per 128-request block
  int lz;           // logits tensor map: z coordinate = request, y = step slot
};

// 16-byte granule g of row r in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw128(int r, int g) { return uint32_t(r) * kTcRowBytes + (uint32_t(g ^ (r & 7)) << 4); }

// The A operand E[r, :] = W1[x(r), :] of a 128-row block in the canonical
// K-major 128-byte-swizzle layout (nkc chunks of [128 rows][128 B]), written by
// the 256 threads tid < 256: thread tid takes row tid % 128 and half tid / 128
// of its 16-byte granules, all issued as asynchronous copies before one wait
// (x < 0: a zero row).  The caller fences for the tensor core afterwards.
static_assert(kTcEpiWarps * 32 == 2 * kTcBM, "gather_w1_rows: two threads per row");
__device__ __forceinline__ void gather_w1_rows(uint8_t* sE, const uint16_t* W1, int rank, int nkc, int tid, int x) {
  const int r = tid & (kTcBM - 1), h = tid / kTcBM;
  const int half = nkc * 4;                       // granules per thread: half of the row's rank / 8
  for (int gi = h * half; gi < (h + 1) * half; ++gi) {
    uint8_t* dst = sE + size_t(gi >> 3) * (kTcBM * kTcRowBytes) + sw128(r, gi & 7);
    if (x >= 0) cp_async16(dst, W1 + size_t(x) * rank + gi * 8);
    else *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
  }
  cp_async_commit();
  cp_async_wait_all();
}

template <int NS>
__global__ void __launch_bounds__(kTcThreads, 1)
    markov_tc_kernel(const __grid_constant__ CUtensorMap tmap_w2, const __grid_constant__ CUtensorMap tmap_u,
                     const __grid_constant__ CUtensorMap tmap_l, MarkovTcArgs ta) {
  const MarkovArgs& a = ta.m;
  extern __shared__ uint8_t s_raw[];
  __shared__ __align__(8) uint64_t bar_full[NS], bar_empty[NS], bar_tfull[2], bar_tempty[2], bar_ufull[NS],
      bar_uempty[NS], bar_done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_err;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(s_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sE = smem;                               // [rank chunk][128 rows][128 B]
  uint8_t* sB = sE + kTcSmemE;                      // [stage][rank][128 B]: W2[k, n0 .. n0+64)
  uint8_t* sU = sB + NS * kTcStageB;                // [stage][128 rows][128 B]  (64 bf16 per row)
  uint8_t* sL = sU + NS * kTcStageU;                // [warp][2 halves][32 rows][128 B]  (32 floats per row)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mb = blockIdx.x / ta.per_mb, j0 = blockIdx.x - (blockIdx.x / ta.per_mb) * ta.per_mb;
  const int row0 = mb * kTcBM;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], 1);
      mbar_init(&bar_ufull[i], 1);
      mbar_init(&bar_uempty[i], 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_tfull[i], 1);
      mbar_init(&bar_tempty[i], 4);
    }
    mbar_init(&bar_done, 1);
    s_err = 0;
    fence_mbar_init();
  }
  if (warp == kTcEpiWarps + 1) tc::tmem_alloc(&s_tmem, kTcTmemCols);
  pdl_wait_primary();                      // the previous step's tokens are complete
  // the error word is reset once per call, after the work before it completes
  if (a.k == 1 && blockIdx.x == 0 && threadIdx.x == 0) *reinterpret_cast<int*>(a.workspace) = 0;
  if (warp < kTcEpiWarps) {
    // A operand: E[r, :] = W1[x_{k-1}(r), :] for this CTA's 128 rows
    {
      const int req = row0 + (threadIdx.x & (kTcBM - 1));
      int x = -1;
      if (req < a.R) {
        x = prev_token(a, req);
        if (x < 0 || x >= a.V) x = -1;
      }
      gather_w1_rows(sE, a.W1, a.rank, ta.nkc, threadIdx.x, x);
    }
    tc::fence_proxy_async_smem();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;

  if (warp == kTcEpiWarps) {
    // ---- TMA producer: W2[:, t*64 .. +64) (MMA operand) and U_k[rows, t*64 .. +64) (epilogue)
    if (lane == 0) {
      // W2 is read by every step: keep it in L2 ahead of U, which is read once
      const uint64_t keep = tc::policy_evict_last(), stream_once = tc::policy_evict_first();
      int i = 0;
      for (int t = j0; t < ta.ntiles; t += ta.per_mb, ++i) {
        const int s = i % NS;
        const uint32_t fresh = ((i / NS) & 1) ^ 1;
        if (!mbar_wait_parity(&bar_empty[s], fresh, kTcMaxPolls)) { s_err = 1; break; }
        mbar_arrive_expect_tx(&bar_full[s], uint32_t(ta.nkc) * 64 * kTcRowBytes);
        for (int kc = 0; kc < ta.nkc; ++kc)     // 64 k-rows of 64 columns per box
          tc::tma_load_2d_hint(sB + size_t(s) * kTcStageB + size_t(kc) * (64 * kTcRowBytes), &tmap_w2, t * kTcBN,
                               kc * 64, &bar_full[s], keep);
        if (!mbar_wait_parity(&bar_uempty[s], fresh, kTcMaxPolls)) { s_err = 1; break; }
        mbar_arrive_expect_tx(&bar_ufull[s], kTcBM * kTcRowBytes);
        tc::tma_load_3d_hint(sU + size_t(s) * kTcStageU, &tmap_u, t * kTcBN, a.k - 1, row0, &bar_ufull[s],
                             stream_once);
      }
      // every issued copy has landed before the CTA may leave
      for (int d = (i >= NS ? i - NS : 0); d < i; ++d) {
        if (!mbar_wait_parity(&bar_full[d % NS], (d / NS) & 1, kTcMaxPolls)) s_err = 1;
        if (!mbar_wait_parity(&bar_ufull[d % NS], (d / NS) & 1, kTcMaxPolls)) s_err = 1;
      }
    }
  } else if (warp == kTcEpiWarps + 1) {
    // ---- MMA issuer
    if (lane == 0) {
      // Descriptors are linear in their 14-bit start-address field (address / 16),
      // so each MMA's descriptor is a base plus a constant: A chunk kc at
      // +kc * 16 KB, 32-byte K step inside a 128-byte row; B k-group kk at
      // +kk * 2 KB.  Computing them once keeps the issue loop short.
      const uint64_t da0 = tc::smem_desc_k_sw128(smem_addr(sE));
      uint64_t db0[NS];
#pragma unroll
      for (int st = 0; st < NS; ++st) db0[st] = tc::smem_desc_mn_sw128(smem_addr(sB) + uint32_t(st) * kTcStageB, 1024, 64 * 64 * 2);
      int i = 0;
      for (int t = j0; t < ta.ntiles; t += ta.per_mb, ++i) {
        const int s = i % NS, tb = i & 1;         // W2 stage, TMEM accumulator buffer
        if (!mbar_wait_parity(&bar_tempty[tb], ((i >> 1) & 1) ^ 1, kTcMaxPolls) ||
            !mbar_wait_parity(&bar_full[s], (i / NS) & 1, kTcMaxPolls)) {
          s_err = 1;
          break;
        }
        tc::fence_after_sync();
        uint64_t dbs = db0[0];
#pragma unroll
        for (int st = 1; st < NS; ++st)
          if (s == st) dbs = db0[st];
        const uint32_t dtm = tmem + uint32_t(tb * kTcBN);
        for (int kk = 0; kk < ta.nkc * 4; ++kk) {
          // A: chunk kk / 4 (16 KB apart), 32-byte K step; B: 16 k-rows = two 1024-byte groups further along K
          const uint64_t da = da0 + uint64_t((kk >> 2) * (kTcBM * kTcRowBytes / 16) + (kk & 3) * 2);
          const uint64_t db = dbs + uint64_t(kk * (2048 / 16));
          tc::mma_bf16(dtm, da, db, kTcIdesc, kk > 0 ? 1u : 0u);
        }
        tc::commit(&bar_empty[s]);            // the W2 stage is free once these MMAs have read it
        tc::commit(&bar_tfull[tb]);           // the accumulator is ready for the epilogue
      }
      tc::commit(&bar_done);
      if (!mbar_wait_parity(&bar_done, 0, kTcMaxPolls)) s_err = 1;
    }
  } else {
    // ---- epilogue group g = warp / 4 takes tiles i = g, g + 2, ...; thread = request row
    const int g = warp >> 2, qd = warp & 3;
    const int rl = qd * 32 + lane;                  // row inside the 128-request block
    const int r = row0 + rl;
    const bool rv = r < a.R;
    const uint64_t keep_part = tc::policy_evict_last();
    uint8_t* stage = sL + size_t(warp) * (2 * 32 * kTcRowBytes);
    int i = g;
    for (int t = j0 + g * ta.per_mb; t < ta.ntiles; t += 2 * ta.per_mb, i += 2) {
      const int n0 = t * kTcBN;
      const int us = i % NS;                        // U stage of tile i (its accumulator buffer is g)
      // warp-uniform outcome: tcgen05.ld below needs all 32 lanes
      if (!__all_sync(0xffffffffu, mbar_wait_parity(&bar_tfull[g], (i >> 1) & 1, kTcMaxPolls) &&
                                       mbar_wait_parity(&bar_ufull[us], (i / NS) & 1, kTcMaxPolls))) {
        s_err = 1;
        break;
      }
      tc::fence_after_sync();
      float acc0[32], acc1[32];
      const uint32_t taddr = tmem + (uint32_t(qd * 32) << 16) + uint32_t(g * kTcBN);
      tc::tmem_ld32(taddr, acc0);
      tc::tmem_ld32(taddr + 32, acc1);
      tc::tmem_ld_wait();
      uint4 u[8];
      const uint8_t* urow = sU + size_t(us) * kTcStageU;
#pragma unroll
      for (int c = 0; c < 8; ++c) u[c] = *reinterpret_cast<const uint4*>(urow + sw128(rl, c));
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_tempty[g]);
      float L[64];
      chunk_logits(u, acc0, acc1, a.logits_bf16 != 0, L);
      // release the U stage only after the adds above consumed its values
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_uempty[us]);
      if (n0 + 64 > a.V) {                          // the last tile: columns past V read -inf
#pragma unroll
        for (int j = 0; j < 64; ++j)
          if (n0 + j >= a.V) L[j] = neg_inf();
      }
      // logits: this warp's 32 rows x 64 columns through swizzled staging, then TMA stores
      if (NS == 2 && a.logits != nullptr) {          // the staging exists only in the two-stage layout
        if (lane == 0) tc::bulk_wait_read_all();     // the previous tile's stores have read the staging
        __syncwarp();
        if (a.logits_bf16) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint4 o;
            o.x = (__float_as_uint(L[8 * c + 0]) >> 16) | (__float_as_uint(L[8 * c + 1]) & 0xFFFF0000u);
            o.y = (__float_as_uint(L[8 * c + 2]) >> 16) | (__float_as_uint(L[8 * c + 3]) & 0xFFFF0000u);
            o.z = (__float_as_uint(L[8 * c + 4]) >> 16) | (__float_as_uint(L[8 * c + 5]) & 0xFFFF0000u);
            o.w = (__float_as_uint(L[8 * c + 6]) >> 16) | (__float_as_uint(L[8 * c + 7]) & 0xFFFF0000u);
            *reinterpret_cast<uint4*>(stage + sw128(lane, c)) = o;
          }
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c)
            *reinterpret_cast<float4*>(stage + (c >> 3) * (32 * kTcRowBytes) + sw128(lane, c & 7)) =
                make_float4(L[4 * c], L[4 * c + 1], L[4 * c + 2], L[4 * c + 3]);
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int z = row0 + qd * 32;
          if (a.logits_bf16) {
            tc::tma_store_3d(&tmap_l, n0, ta.lz, z, stage);
          } else {
            tc::tma_store_3d(&tmap_l, n0, ta.lz, z, stage);
            tc::tma_store_3d(&tmap_l, n0 + 32, ta.lz, z, stage + 32 * kTcRowBytes);
          }
          tc::bulk_commit();
        }
      }
      if (!rv) continue;
      store_part(a.part + size_t(r) * a.ntile + t, chunk_partial(L, n0, a), keep_part);
    }
    if (NS == 2 && lane == 0 && a.logits != nullptr) tc::bulk_wait_all();   // logits written before the sampler reads them
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kTcEpiWarps + 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTcTmemCols);
  }
  if (threadIdx.x == 0 && s_err) record_device_error(a.workspace, SPECV_ERR_TIMEOUT);
  pdl_launch_dependents();   // measured: triggering at the start instead was slower
}

// ---------------------------------------------------------------------------
// Wide tensor-core form for drafting without kept logits: N = 256 columns per
// MMA.  At N = 64 each tcgen05.mma re-reads a 4 KB slice of the A operand from
// shared memory for 2 KB of B, and the operand reads bound the tensor core;
// at N = 256 one A read serves four times the columns.
//   W2 ring: stages of one 64-row rank chunk of a 256-column tile (four 8 KB
//            TMA boxes, 32 KB), filled by the W2 TMA warp;
//   U rings: one per epilogue group, two 64-column chunks of U (16 KB
//            each), each filled by its own TMA warp, so U never waits behind
//            W2.  A ring is waited on only by the group that empties it, so a
//            waiter is never two phases ahead of a slot (a parity wait cannot
//            tell phase n from phase n + 2);
//   MMA:     four K = 16 instructions per rank chunk into one of two
//            256-column TMEM accumulators;
//   epilogue: two groups of four warps alternate tiles; each reads its
//            accumulator in four 64-column chunks, adds U and writes the
//            64-column tile partials the sampler combines (tile_w = 64).
constexpr int kWN = 256;                  // columns per tile (UMMA N)
constexpr int kWChunks = kWN / 64;        // 64-column chunks per tile
constexpr int kWStagesB = 3;              // W2 ring: rank chunks
constexpr int kWStagesU = 2;              // U ring per epilogue group: 64-column chunks
constexpr int kWThreads = (kTcEpiWarps + 4) * 32;    // + W2 TMA, two U TMA, MMA warps
constexpr uint32_t kWTmemCols = 512;      // two accumulator buffers of 256 columns
constexpr size_t kWStageB = size_t(kWChunks) * 64 * kTcRowBytes;       // 32 KB
constexpr size_t kWStageU = size_t(kTcBM) * kTcRowBytes;               // 16 KB
constexpr size_t kWSmem = kTcSmemE + kWStagesB * kWStageB + 2 * kWStagesU * kWStageU + 1024;
constexpr uint32_t kWIdesc = tc::idesc_bf16_f32(kTcBM, kWN, true);     // B = W2, MN-major

__global__ void __launch_bounds__(kWThreads, 1)
    markov_tcw_kernel(const __grid_constant__ CUtensorMap tmap_w2, const __grid_constant__ CUtensorMap tmap_u,
                      const __grid_constant__ CUtensorMap tmap_l, MarkovTcArgs ta) {
  const MarkovArgs& a = ta.m;
  extern __shared__ uint8_t s_raw[];
  __shared__ __align__(8) uint64_t bar_full[kWStagesB], bar_empty[kWStagesB], bar_ufull[2][kWStagesU],
      bar_uempty[2][kWStagesU], bar_tfull[2], bar_tempty[2], bar_done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_err;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(s_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sE = smem;                               // [rank chunk][128 rows][128 B]
  uint8_t* sB = sE + kTcSmemE;                      // [stage][column block][64 k-rows][128 B]
  uint8_t* sU = sB + kWStagesB * kWStageB;          // [group][stage][128 rows][128 B]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mb = blockIdx.x / ta.per_mb, j0 = blockIdx.x - (blockIdx.x / ta.per_mb) * ta.per_mb;
  const int row0 = mb * kTcBM;
  const int nwt = (ta.ntiles + kWChunks - 1) / kWChunks;       // 256-column tiles

  if (threadIdx.x == 0) {
    for (int i = 0; i < kWStagesB; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], 1);
    }
    for (int g = 0; g < 2; ++g)
      for (int i = 0; i < kWStagesU; ++i) {
        mbar_init(&bar_ufull[g][i], 1);
        mbar_init(&bar_uempty[g][i], 4);
      }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_tfull[i], 1);
      mbar_init(&bar_tempty[i], 4);
    }
    mbar_init(&bar_done, 1);
    s_err = 0;
    fence_mbar_init();
  }
  if (warp == kTcEpiWarps + 3) tc::tmem_alloc(&s_tmem, kWTmemCols);
  pdl_wait_primary();                      // the previous step's tokens are complete
  // the error word is reset once per call, after the work before it completes
  if (a.k == 1 && blockIdx.x == 0 && threadIdx.x == 0) *reinterpret_cast<int*>(a.workspace) = 0;
  if (warp < kTcEpiWarps) {
    // A operand: E[r, :] = W1[x_{k-1}(r), :] for this CTA's 128 rows
    {
      const int req = row0 + (threadIdx.x & (kTcBM - 1));
      int x = -1;
      if (req < a.R) {
        x = prev_token(a, req);
        if (x < 0 || x >= a.V) x = -1;
      }
      gather_w1_rows(sE, a.W1, a.rank, ta.nkc, threadIdx.x, x);
    }
    tc::fence_proxy_async_smem();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;

  if (warp == kTcEpiWarps) {
    // ---- W2 producer: one stage per (tile, rank chunk), four 64-column boxes
    if (lane == 0) {
      const uint64_t keep = tc::policy_evict_last();
      int q = 0;                                   // (tile, chunk) sequence number
      for (int t = j0; t < nwt; t += ta.per_mb)
        for (int kc = 0; kc < ta.nkc; ++kc, ++q) {
          const int s = q % kWStagesB;
          if (!mbar_wait_parity(&bar_empty[s], ((q / kWStagesB) & 1) ^ 1, kTcMaxPolls)) { s_err = 1; t = nwt; break; }
          mbar_arrive_expect_tx(&bar_full[s], uint32_t(kWStageB));
          for (int b = 0; b < kWChunks; ++b)
            tc::tma_load_2d_hint(sB + size_t(s) * kWStageB + size_t(b) * (64 * kTcRowBytes), &tmap_w2,
                                 t * kWN + b * 64, kc * 64, &bar_full[s], keep);
        }
      for (int d = (q >= kWStagesB ? q - kWStagesB : 0); d < q; ++d)   // issued copies have landed
        if (!mbar_wait_parity(&bar_full[d % kWStagesB], (d / kWStagesB) & 1, kTcMaxPolls)) s_err = 1;
    }
  } else if (warp == kTcEpiWarps + 1 || warp == kTcEpiWarps + 2) {
    // ---- U producer of epilogue group g: 64-column chunks of U_k for its tiles
    const int g = warp - (kTcEpiWarps + 1);
    if (lane == 0) {
      const uint64_t once = tc::policy_evict_first();
      uint8_t* ring = sU + size_t(g) * kWStagesU * kWStageU;
      int q = 0;                                   // chunk sequence number within the group
      for (int t = j0 + g * ta.per_mb; t < nwt; t += 2 * ta.per_mb)
        for (int c = 0; c < kWChunks; ++c, ++q) {
          const int s = q % kWStagesU;
          if (!mbar_wait_parity(&bar_uempty[g][s], ((q / kWStagesU) & 1) ^ 1, kTcMaxPolls)) { s_err = 1; t = nwt; break; }
          mbar_arrive_expect_tx(&bar_ufull[g][s], uint32_t(kWStageU));
          tc::tma_load_3d_hint(ring + size_t(s) * kWStageU, &tmap_u, t * kWN + c * 64, a.k - 1, row0,
                               &bar_ufull[g][s], once);
        }
      for (int d = (q >= kWStagesU ? q - kWStagesU : 0); d < q; ++d)
        if (!mbar_wait_parity(&bar_ufull[g][d % kWStagesU], (d / kWStagesU) & 1, kTcMaxPolls)) s_err = 1;
    }
  } else if (warp == kTcEpiWarps + 3) {
    // ---- MMA issuer
    if (lane == 0) {
      const uint64_t da0 = tc::smem_desc_k_sw128(smem_addr(sE));
      uint64_t db0[kWStagesB];
#pragma unroll
      for (int st = 0; st < kWStagesB; ++st)
        db0[st] = tc::smem_desc_mn_sw128(smem_addr(sB) + uint32_t(st) * uint32_t(kWStageB), 1024, 64 * kTcRowBytes);
      int q = 0, i = 0;
      bool ok = true;
      for (int t = j0; t < nwt && ok; t += ta.per_mb, ++i) {
        const int tb = i & 1;
        if (!mbar_wait_parity(&bar_tempty[tb], ((i >> 1) & 1) ^ 1, kTcMaxPolls)) { s_err = 1; break; }
        tc::fence_after_sync();
        const uint32_t dtm = tmem + uint32_t(tb * kWN);
        for (int kc = 0; kc < ta.nkc; ++kc, ++q) {
          const int s = q % kWStagesB;
          if (!mbar_wait_parity(&bar_full[s], (q / kWStagesB) & 1, kTcMaxPolls)) { s_err = 1; ok = false; break; }
          tc::fence_after_sync();
          uint64_t dbs = db0[0];
#pragma unroll
          for (int st = 1; st < kWStagesB; ++st)
            if (s == st) dbs = db0[st];
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // A: chunk kc (16 KB apart), 32-byte K step; B: 16 k-rows = two 1024-byte groups
            const uint64_t da = da0 + uint64_t(kc * (kTcBM * kTcRowBytes / 16) + kk * 2);
            const uint64_t db = dbs + uint64_t(kk * (2048 / 16));
            tc::mma_bf16(dtm, da, db, kWIdesc, (kc > 0 || kk > 0) ? 1u : 0u);
          }
          tc::commit(&bar_empty[s]);          // the W2 stage is free once these MMAs have read it
        }
        if (ok) tc::commit(&bar_tfull[tb]);   // the accumulator is ready for the epilogue
      }
      tc::commit(&bar_done);
      if (!mbar_wait_parity(&bar_done, 0, kTcMaxPolls)) s_err = 1;
    }
  } else {
    // ---- epilogue group g = warp / 4 takes tiles i = g, g + 2, ...; thread = request row
    const int g = warp >> 2, qd = warp & 3;
    const int rl = qd * 32 + lane;
    const int r = row0 + rl;
    const bool rv = r < a.R;
    const uint64_t keep_part = tc::policy_evict_last();
    uint8_t* ring = sU + size_t(g) * kWStagesU * kWStageU;
    int i = g;
    for (int t = j0 + g * ta.per_mb; t < nwt; t += 2 * ta.per_mb, i += 2) {
      if (!__all_sync(0xffffffffu, mbar_wait_parity(&bar_tfull[g], (i >> 1) & 1, kTcMaxPolls))) {
        s_err = 1;
        break;
      }
      tc::fence_after_sync();
      bool ok = true;
      for (int c = 0; c < kWChunks; ++c) {
        const int q = (i >> 1) * kWChunks + c, us = q % kWStagesU;   // this group's chunk sequence
        float acc0[32], acc1[32];
        const uint32_t taddr = tmem + (uint32_t(qd * 32) << 16) + uint32_t(g * kWN + c * 64);
        tc::tmem_ld32(taddr, acc0);
        tc::tmem_ld32(taddr + 32, acc1);
        tc::tmem_ld_wait();
        if (c == kWChunks - 1) {               // the accumulator has been read
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_tempty[g]);
        }
        if (!__all_sync(0xffffffffu, mbar_wait_parity(&bar_ufull[g][us], (q / kWStagesU) & 1, kTcMaxPolls))) {
          s_err = 1;
          ok = false;
          break;
        }
        uint4 u[8];
        const uint8_t* urow = ring + size_t(us) * kWStageU;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) u[cc] = *reinterpret_cast<const uint4*>(urow + sw128(rl, cc));
        const int n0 = t * kWN + c * 64;
        float L[64];
        chunk_logits(u, acc0, acc1, a.logits_bf16, L);
        if (a.logits != nullptr) {
          // bf16 logits kept: this warp's 32 rows of the chunk go out through its
          // own 4 KB part of the U slot (its values are consumed), in the
          // 128-byte swizzle the TMA store expects, one 64-column box.
          uint8_t* wst = const_cast<uint8_t*>(urow) + size_t(qd) * 32 * kTcRowBytes;
          __syncwarp();
          const int z = row0 + qd * 32;
          if (a.logits_bf16) {                   // (float32 logits are stored by markov_tc_kernel)
#pragma unroll
            for (int cc = 0; cc < 8; ++cc)
              *reinterpret_cast<uint4*>(wst + sw128(lane, cc)) =
                  make_uint4((__float_as_uint(L[8 * cc + 0]) >> 16) | (__float_as_uint(L[8 * cc + 1]) & 0xFFFF0000u),
                             (__float_as_uint(L[8 * cc + 2]) >> 16) | (__float_as_uint(L[8 * cc + 3]) & 0xFFFF0000u),
                             (__float_as_uint(L[8 * cc + 4]) >> 16) | (__float_as_uint(L[8 * cc + 5]) & 0xFFFF0000u),
                             (__float_as_uint(L[8 * cc + 6]) >> 16) | (__float_as_uint(L[8 * cc + 7]) & 0xFFFF0000u));
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tc::tma_store_3d(&tmap_l, n0, ta.lz, z, wst);
              tc::bulk_commit();
            }
          }
        }
        if (n0 + 64 > a.V) {
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (n0 + j >= a.V) L[j] = neg_inf();
        }
        MarkovPart mp;
        const bool wp = rv && n0 < a.V;
        if (wp) mp = chunk_partial(L, n0, a);
        // The slot is released only now: the adds above consumed every value
        // read from it, and the store has read what was staged in it (waited
        // for after the partial, which overlaps the store's read), so no read
        // can still be outstanding when the copy of a later chunk overwrites it.
        if (a.logits != nullptr && lane == 0) tc::bulk_wait_read_all();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_uempty[g][us]);
        if (wp) store_part(a.part + size_t(r) * a.ntile + (n0 >> 6), mp, keep_part);
      }
      if (!ok) break;
    }
    if (lane == 0 && a.logits != nullptr) tc::bulk_wait_all();   // logits written before the sampler reads them
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kTcEpiWarps + 3) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kWTmemCols);
  }
  if (threadIdx.x == 0 && s_err) record_device_error(a.workspace, SPECV_ERR_TIMEOUT);
  pdl_launch_dependents();   // measured: triggering at the start instead was slower
}

// ---------------------------------------------------------------------------
// markov_tc2: the same step on CTA pairs.  A cluster of two CTAs (two SMs)
// owns two 128-request blocks, one per CTA, and a strided set of 256-column
// tiles.  One thread of the even CTA issues tcgen05.mma.cta_group::2 with
// M = 256 (each CTA contributes the W1 rows of its own block), N = 256 and
// K = 16, so each CTA stages only its half of every W2 tile (128 columns):
// half the W2 bytes per SM of markov_tcw and twice the ring stages in the same
// shared memory.  Each CTA's tensor memory holds its own 128 accumulator rows;
// its epilogue is markov_tcw's without logit stores: this is the form for
// drafting that keeps no logits (with kept logits the step is bound by their
// DRAM writes and markov_tcw / markov_tc are as fast).
//
// Cross-CTA protocol: each CTA's W2 copies complete on the even CTA's full
// barrier (which expects both halves); the MMA commits arrive on the empty and
// accumulator-full barriers of both CTAs; both CTAs' epilogue warps arrive on
// the even CTA's accumulator-empty barrier.  Every wait is bounded, each CTA
// waits until the last commits aimed at it have arrived, and a cluster barrier
// precedes exit, so no copy or arrival targets a CTA that has exited.
// TN: columns per tile (the MMA's N).  The tensor memory's 512 columns hold
// 512 / TN accumulators; each CTA stages TN / 2 W2 columns per rank chunk in a
// ring of 64 KB.
template <int TN>
struct PairShape {
  static constexpr int kChunks = TN / 64;                               // 64-column chunks per tile
  static constexpr int kAcc = 512 / TN;                                 // accumulators
  static constexpr int kPN = TN / 2;                                    // W2 columns per CTA per tile
  static constexpr size_t kStageB = size_t(kPN / 64) * 64 * kTcRowBytes;   // one rank chunk of them
  static constexpr int kStages = int(64 * 1024 / kStageB);
  static constexpr uint32_t kIdesc = tc::idesc_bf16_f32(2 * kTcBM, TN, true);   // M = 256 over the pair, B MN-major
};
constexpr int kPStagesU = 3;     // U chunks in flight per epilogue group (the epilogue sets the pace)
constexpr size_t kPSmem = kTcSmemE + 64 * 1024 + 2 * kPStagesU * kWStageU + 1024;

template <int TN>
__global__ void __launch_bounds__(kWThreads, 1)
    markov_tc2_kernel(const __grid_constant__ CUtensorMap tmap_w2, const __grid_constant__ CUtensorMap tmap_u,
                      MarkovTcArgs ta) {
  using PS = PairShape<TN>;
  constexpr int NS = PS::kStages, NACC = PS::kAcc, NCH = PS::kChunks;
  const MarkovArgs& a = ta.m;
  extern __shared__ uint8_t s_raw[];
  __shared__ __align__(8) uint64_t bar_full[NS], bar_empty[NS], bar_ufull[2][kPStagesU], bar_uempty[2][kPStagesU],
      bar_tfull[NACC], bar_tempty[NACC], bar_done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_err;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(s_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sE = smem;                               // [rank chunk][128 rows][128 B]
  uint8_t* sB = sE + kTcSmemE;                      // [stage][column block][64 k-rows][128 B]
  uint8_t* sU = sB + NS * PS::kStageB;              // [group][stage][128 rows][128 B]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int crank = int(cluster_ctarank());         // 0: issues the pair MMAs
  const int cl = int(blockIdx.x >> 1);
  const int pb = cl / ta.per_mb, j0 = cl - pb * ta.per_mb;
  const int row0 = (2 * pb + crank) * kTcBM;
  const int nwt = (ta.ntiles + NCH - 1) / NCH;                 // TN-column tiles

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], 1);
    }
    for (int g = 0; g < 2; ++g)
      for (int i = 0; i < kPStagesU; ++i) {
        mbar_init(&bar_ufull[g][i], 1);
        mbar_init(&bar_uempty[g][i], 4);
      }
    for (int i = 0; i < NACC; ++i) {
      mbar_init(&bar_tfull[i], 1);
      mbar_init(&bar_tempty[i], 2 * 4);          // four epilogue warps of each CTA
    }
    mbar_init(&bar_done, 1);
    s_err = 0;
    fence_mbar_init();
  }
  if (warp == kTcEpiWarps + 3) tc::tmem_alloc_pair(&s_tmem, kWTmemCols);
  pdl_wait_primary();                      // the previous step's tokens are complete
  // the error word is reset once per call, after the work before it completes
  if (a.k == 1 && blockIdx.x == 0 && threadIdx.x == 0) *reinterpret_cast<int*>(a.workspace) = 0;
  if (warp < kTcEpiWarps) {
    // A operand: E[r, :] = W1[x_{k-1}(r), :] for this CTA's 128 rows
    {
      const int req = row0 + (threadIdx.x & (kTcBM - 1));
      int x = -1;
      if (req < a.R) {
        x = prev_token(a, req);
        if (x < 0 || x >= a.V) x = -1;
      }
      gather_w1_rows(sE, a.W1, a.rank, ta.nkc, threadIdx.x, x);
    }
    tc::fence_proxy_async_smem();
  }
  // Both CTAs' barriers are initialised and both A halves written before any
  // copy, arrival or MMA crosses to the other CTA.
  tc::fence_before_sync();
  __syncwarp();
  cluster_arrive_release();
  cluster_wait_acquire();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;

  if (warp == kTcEpiWarps) {
    // ---- W2 producer: this CTA's TN / 2 columns of one (tile, rank chunk) per stage
    if (lane == 0) {
      const uint64_t keep = tc::policy_evict_last();
      int q = 0;                                   // (tile, chunk) sequence number
      for (int t = j0; t < nwt; t += ta.per_mb)
        for (int kc = 0; kc < ta.nkc; ++kc, ++q) {
          const int s = q % NS;
          if (!mbar_wait_parity(&bar_empty[s], ((q / NS) & 1) ^ 1, kTcMaxPolls)) { s_err = 1; t = nwt; break; }
          if (crank == 0) mbar_arrive_expect_tx(&bar_full[s], uint32_t(2 * PS::kStageB));
          const uint32_t full0 = cluster_map_shared(&bar_full[s], 0);
          for (int b = 0; b < PS::kPN / 64; ++b)
            tc::tma_load_2d_pair(sB + size_t(s) * PS::kStageB + size_t(b) * (64 * kTcRowBytes), &tmap_w2,
                                 t * TN + crank * PS::kPN + b * 64, kc * 64, full0, keep);
        }
      // the MMAs that read the last stages have completed, and their commits
      // to this CTA have arrived
      for (int d = (q >= NS ? q - NS : 0); d < q; ++d)
        if (!mbar_wait_parity(&bar_empty[d % NS], (d / NS) & 1, kTcMaxPolls)) s_err = 1;
    }
  } else if (warp == kTcEpiWarps + 1 || warp == kTcEpiWarps + 2) {
    // ---- U producer of epilogue group g: 64-column chunks of this CTA's U_k rows
    const int g = warp - (kTcEpiWarps + 1);
    if (lane == 0) {
      const uint64_t once = tc::policy_evict_first();
      uint8_t* ring = sU + size_t(g) * kPStagesU * kWStageU;
      int q = 0;
      for (int t = j0 + g * ta.per_mb; t < nwt; t += 2 * ta.per_mb)
        for (int c = 0; c < NCH; ++c, ++q) {
          const int s = q % kPStagesU;
          if (!mbar_wait_parity(&bar_uempty[g][s], ((q / kPStagesU) & 1) ^ 1, kTcMaxPolls)) { s_err = 1; t = nwt; break; }
          mbar_arrive_expect_tx(&bar_ufull[g][s], uint32_t(kWStageU));
          tc::tma_load_3d_hint(ring + size_t(s) * kWStageU, &tmap_u, t * TN + c * 64, a.k - 1, row0,
                               &bar_ufull[g][s], once);
        }
      for (int d = (q >= kPStagesU ? q - kPStagesU : 0); d < q; ++d)
        if (!mbar_wait_parity(&bar_ufull[g][d % kPStagesU], (d / kPStagesU) & 1, kTcMaxPolls)) s_err = 1;
    }
  } else if (warp == kTcEpiWarps + 3) {
    // ---- pair MMA issuer (even CTA)
    if (lane == 0 && crank == 0) {
      const uint64_t da0 = tc::smem_desc_k_sw128(smem_addr(sE));
      const uint64_t db0 = tc::smem_desc_mn_sw128(smem_addr(sB), 1024, 64 * kTcRowBytes);
      int q = 0, i = 0;
      bool ok = true;
      for (int t = j0; t < nwt && ok; t += ta.per_mb, ++i) {
        const int tb = i % NACC;                   // accumulator
        if (!mbar_wait_parity(&bar_tempty[tb], ((i / NACC) & 1) ^ 1, kTcMaxPolls)) { s_err = 1; break; }
        tc::fence_after_sync();
        const uint32_t dtm = tmem + uint32_t(tb * TN);
        for (int kc = 0; kc < ta.nkc; ++kc, ++q) {
          const int s = q % NS;
          if (!mbar_wait_parity(&bar_full[s], (q / NS) & 1, kTcMaxPolls)) { s_err = 1; ok = false; break; }
          tc::fence_after_sync();
          const uint64_t dbs = db0 + uint64_t(s) * (PS::kStageB / 16);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // A: chunk kc (16 KB apart), 32-byte K step; B: 16 k-rows = two 1024-byte groups
            const uint64_t da = da0 + uint64_t(kc * (kTcBM * kTcRowBytes / 16) + kk * 2);
            const uint64_t db = dbs + uint64_t(kk * (2048 / 16));
            tc::mma_bf16_pair(dtm, da, db, PS::kIdesc, (kc > 0 || kk > 0) ? 1u : 0u);
          }
          tc::commit_pair(&bar_empty[s], 0x3);    // both CTAs' stage s is free once these MMAs have read it
        }
        if (ok) tc::commit_pair(&bar_tfull[tb], 0x3);   // both accumulator halves are ready
      }
      tc::commit_pair(&bar_done, 0x1);
      if (!mbar_wait_parity(&bar_done, 0, kTcMaxPolls)) s_err = 1;
      // both CTAs' epilogues have released the accumulators of the last tiles
      for (int tb = 0; tb < NACC; ++tb) {
        const int uses = (i + NACC - 1 - tb) / NACC;   // tiles 0 .. i-1 with index % NACC == tb
        if (uses > 0 && !mbar_wait_parity(&bar_tempty[tb], (uses - 1) & 1, kTcMaxPolls)) s_err = 1;
      }
    }
  } else {
    // ---- epilogue group g = warp / 4 takes tiles i = g, g + 2, ... (accumulator
    // i % NACC); thread = request row
    const int g = warp >> 2, qd = warp & 3;
    const int rl = qd * 32 + lane;
    const int r = row0 + rl;
    const bool rv = r < a.R;
    const uint64_t keep_part = tc::policy_evict_last();
    uint8_t* ring = sU + size_t(g) * kPStagesU * kWStageU;
    int i = g;
    for (int t = j0 + g * ta.per_mb; t < nwt; t += 2 * ta.per_mb, i += 2) {
      const int tb = i % NACC;
      if (!__all_sync(0xffffffffu, mbar_wait_parity(&bar_tfull[tb], (i / NACC) & 1, kTcMaxPolls))) {
        s_err = 1;
        break;
      }
      tc::fence_after_sync();
      bool ok = true;
      for (int c = 0; c < NCH; ++c) {
        const int q = (i >> 1) * NCH + c, us = q % kPStagesU;   // this group's chunk sequence
        float acc0[32], acc1[32];
        const uint32_t taddr = tmem + (uint32_t(qd * 32) << 16) + uint32_t(tb * TN + c * 64);
        tc::tmem_ld32(taddr, acc0);
        tc::tmem_ld32(taddr + 32, acc1);
        tc::tmem_ld_wait();
        if (c == NCH - 1) {                    // this CTA's half of the accumulator has been read
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(cluster_map_shared(&bar_tempty[tb], 0));
        }
        if (!__all_sync(0xffffffffu, mbar_wait_parity(&bar_ufull[g][us], (q / kPStagesU) & 1, kTcMaxPolls))) {
          s_err = 1;
          ok = false;
          break;
        }
        uint4 u[8];
        const uint8_t* urow = ring + size_t(us) * kWStageU;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) u[cc] = *reinterpret_cast<const uint4*>(urow + sw128(rl, cc));
        const int n0 = t * TN + c * 64;
        float L[64];
        chunk_logits(u, acc0, acc1, a.logits_bf16, L);
        // The U slot is released once the adds above have consumed every value
        // read from it, so no read is outstanding when a later copy refills it.
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_uempty[g][us]);
        if (n0 + 64 > a.V) {
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (n0 + j >= a.V) L[j] = neg_inf();
        }
        if (rv && n0 < a.V) store_part(a.part + size_t(r) * a.ntile + (n0 >> 6), chunk_partial(L, n0, a), keep_part);
      }
      if (!ok) break;
    }
  }
  tc::fence_before_sync();
  __syncwarp();
  cluster_arrive_release();
  cluster_wait_acquire();
  if (warp == kTcEpiWarps + 3) {
    tc::fence_after_sync();
    tc::tmem_dealloc_pair(tmem, kWTmemCols);
  }
  if (threadIdx.x == 0 && s_err) record_device_error(a.workspace, SPECV_ERR_TIMEOUT);
  pdl_launch_dependents();   // measured: triggering at the start instead was slower
}

// ---------------------------------------------------------------------------
// Recomputing the draft logits a verification reads.  After drafting without
// kept logits and scheduling, only the rows (r, k) with k < l_r are verified.
// markov_rows_prep lists them; markov_rows_kernel recomputes
// L = U[r, k] + W1[x_{k-1}] . W2 for those rows with the same 256-column
// tensor-core tiling as markov_tcw (so the float32 sums, and their bf16
// rounding, are the ones the draws used) and writes them as bf16 into the
// usual [R, gamma, V] layout.  Rows are gathered, so U comes in by 16-byte
// async copies issued by each epilogue warp for its own 32 rows, two chunks
// ahead, rather than by a TMA box; the logits leave the same way.
constexpr int kRowsListOff = 64;          // workspace header: int32 live-row count at this byte offset
constexpr int kRowsUStages = 2;           // U chunks in flight per epilogue group
constexpr size_t kRowsSmem = kTcSmemE + kWStagesB * kWStageB + size_t(2) * kRowsUStages * kWStageU + 1024;

struct RowsArgs {
  const uint16_t* U;
  const uint16_t* W1;
  const int32_t* anchor;
  const int32_t* tokens;      // [R, gamma]
  const int32_t* lengths;     // [R] or null (gamma)
  uint16_t* out;              // [R, gamma, V] bf16
  int32_t* rows;              // [R * gamma]: r * gamma + k of each live row, in (r, k) order
  void* workspace;
  int R, gamma, V, rank, nkc;
  int ntiles;                 // 256-column tiles
};

// one CTA: prefix over the lengths, then the list of live rows
__global__ void __launch_bounds__(1024) markov_rows_prep(RowsArgs a) {
  __shared__ int s_warp[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = (a.R + 1023) / 1024;
  const int r0 = threadIdx.x * per, r1 = min(a.R, r0 + per);
  int cnt = 0;
  bool bad = false;
  for (int r = r0; r < r1; ++r) {
    int l = a.lengths ? a.lengths[r] : a.gamma;
    if (l < 0 || l > a.gamma) { l = 0; bad = true; }
    cnt += l;
  }
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int wpre = 0, total = 0;
  for (int w = 0; w < 32; ++w) {
    if (w < warp) wpre += s_warp[w];
    total += s_warp[w];
  }
  int off = wpre + incl - cnt;
  for (int r = r0; r < r1; ++r) {
    int l = a.lengths ? a.lengths[r] : a.gamma;
    if (l < 0 || l > a.gamma) l = 0;
    for (int k = 0; k < l; ++k) a.rows[off + k] = r * a.gamma + k;
    off += l;
  }
  if (threadIdx.x == 0) {
    *reinterpret_cast<int*>(a.workspace) = 0;
    reinterpret_cast<int*>(a.workspace)[kRowsListOff / 4] = total;
  }
  __syncthreads();
  if (bad) record_device_error(a.workspace, SPECV_ERR_DEVICE_DATA);
  pdl_launch_dependents();
}

__global__ void __launch_bounds__(kTcThreads, 1)
    markov_rows_kernel(const __grid_constant__ CUtensorMap tmap_w2, RowsArgs a) {
  extern __shared__ uint8_t s_raw[];
  __shared__ __align__(8) uint64_t bar_full[kWStagesB], bar_empty[kWStagesB], bar_tfull[2], bar_tempty[2], bar_done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_err, s_n;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(s_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sE = smem;                               // [rank chunk][128 rows][128 B]
  uint8_t* sB = sE + kTcSmemE;                      // [stage][column block][64 k-rows][128 B]
  uint8_t* sU = sB + kWStagesB * kWStageB;          // [group][stage][128 rows][128 B], each thread its own row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_wait_primary();                               // the row list is complete
  if (threadIdx.x == 0) s_n = reinterpret_cast<const int*>(a.workspace)[kRowsListOff / 4];
  __syncthreads();
  const int n_rows = s_n;
  const int n_mb = (n_rows + kTcBM - 1) / kTcBM;
  if (n_mb == 0) return;                            // block-uniform: nothing to recompute
  const int per_mb = int(gridDim.x) / n_mb > 0 ? int(gridDim.x) / n_mb : 1;
  const int mb = int(blockIdx.x) / per_mb, j0 = int(blockIdx.x) - (int(blockIdx.x) / per_mb) * per_mb;
  if (mb >= n_mb) return;                           // block-uniform: an idle CTA (n_mb * per_mb <= grid)
  const int row0 = mb * kTcBM;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kWStagesB; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_tfull[i], 1);
      mbar_init(&bar_tempty[i], 4);
    }
    mbar_init(&bar_done, 1);
    s_err = 0;
    fence_mbar_init();
  }
  if (warp == kTcEpiWarps + 1) tc::tmem_alloc(&s_tmem, kWTmemCols);
  if (warp < kTcEpiWarps) {
    // A operand: the previous token of each listed row
    {
      const int rl = threadIdx.x & (kTcBM - 1);
      int x = -1;
      if (row0 + rl < n_rows) {
        const int rk = a.rows[row0 + rl];
        const int r = rk / a.gamma, k = rk - (rk / a.gamma) * a.gamma;
        x = k == 0 ? a.anchor[r] : a.tokens[size_t(r) * a.gamma + (k - 1)];
        if (x < 0 || x >= a.V) x = -1;
      }
      gather_w1_rows(sE, a.W1, a.rank, a.nkc, threadIdx.x, x);
    }
    tc::fence_proxy_async_smem();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;

  if (warp == kTcEpiWarps) {
    // ---- W2 producer (as in markov_tcw)
    if (lane == 0) {
      const uint64_t keep = tc::policy_evict_last();
      int q = 0;
      for (int t = j0; t < a.ntiles; t += per_mb)
        for (int kc = 0; kc < a.nkc; ++kc, ++q) {
          const int s = q % kWStagesB;
          if (!mbar_wait_parity(&bar_empty[s], ((q / kWStagesB) & 1) ^ 1, kTcMaxPolls)) { s_err = 1; t = a.ntiles; break; }
          mbar_arrive_expect_tx(&bar_full[s], uint32_t(kWStageB));
          for (int b = 0; b < kWChunks; ++b)
            tc::tma_load_2d_hint(sB + size_t(s) * kWStageB + size_t(b) * (64 * kTcRowBytes), &tmap_w2,
                                 t * kWN + b * 64, kc * 64, &bar_full[s], keep);
        }
      for (int d = (q >= kWStagesB ? q - kWStagesB : 0); d < q; ++d)
        if (!mbar_wait_parity(&bar_full[d % kWStagesB], (d / kWStagesB) & 1, kTcMaxPolls)) s_err = 1;
    }
  } else if (warp == kTcEpiWarps + 1) {
    // ---- MMA issuer (as in markov_tcw)
    if (lane == 0) {
      const uint64_t da0 = tc::smem_desc_k_sw128(smem_addr(sE));
      uint64_t db0[kWStagesB];
#pragma unroll
      for (int st = 0; st < kWStagesB; ++st)
        db0[st] = tc::smem_desc_mn_sw128(smem_addr(sB) + uint32_t(st) * uint32_t(kWStageB), 1024, 64 * kTcRowBytes);
      int q = 0, i = 0;
      bool ok = true;
      for (int t = j0; t < a.ntiles && ok; t += per_mb, ++i) {
        const int tb = i & 1;
        if (!mbar_wait_parity(&bar_tempty[tb], ((i >> 1) & 1) ^ 1, kTcMaxPolls)) { s_err = 1; break; }
        tc::fence_after_sync();
        const uint32_t dtm = tmem + uint32_t(tb * kWN);
        for (int kc = 0; kc < a.nkc; ++kc, ++q) {
          const int s = q % kWStagesB;
          if (!mbar_wait_parity(&bar_full[s], (q / kWStagesB) & 1, kTcMaxPolls)) { s_err = 1; ok = false; break; }
          tc::fence_after_sync();
          uint64_t dbs = db0[0];
#pragma unroll
          for (int st = 1; st < kWStagesB; ++st)
            if (s == st) dbs = db0[st];
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t da = da0 + uint64_t(kc * (kTcBM * kTcRowBytes / 16) + kk * 2);
            const uint64_t db = dbs + uint64_t(kk * (2048 / 16));
            tc::mma_bf16(dtm, da, db, kWIdesc, (kc > 0 || kk > 0) ? 1u : 0u);
          }
          tc::commit(&bar_empty[s]);
        }
        if (ok) tc::commit(&bar_tfull[tb]);
      }
      tc::commit(&bar_done);
      if (!mbar_wait_parity(&bar_done, 0, kTcMaxPolls)) s_err = 1;
    }
  } else {
    // ---- epilogue group g takes tiles i = g, g + 2, ...; thread = listed row.
    // A warp moves its 32 rows' chunks cooperatively: in each 16-byte copy or
    // store instruction lane l takes granule l % 8 of row 4m + l / 8, so one
    // instruction covers four whole 128-byte row pieces instead of 32
    // scattered granules.  The warp's staging holds row j's granule q at
    // granule q ^ (j % 8) (conflict-free both ways); each thread reads its own
    // row from it, and the bf16 logits go back through it to be stored.
    const int g = warp >> 2, qd = warp & 3;
    const int rl = qd * 32 + lane;
    const bool rv = row0 + rl < n_rows;
    int rk = 0;
    if (rv) rk = a.rows[row0 + rl];
    const int gq = lane & 7;                           // granule this lane moves
    int rks[8];                                        // rows 4m + lane / 8 of this warp
    bool vld[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int jr = 4 * m + (lane >> 3);
      rks[m] = __shfl_sync(0xffffffffu, rk, jr);
      vld[m] = row0 + qd * 32 + jr < n_rows;
    }
    uint8_t* wstage = sU + size_t(g * kRowsUStages) * kWStageU + size_t(qd) * 32 * kTcRowBytes;   // + stage * kWStageU
    // this group's chunk sequence: n = (tile index within the group) * 4 + c
    const int n_tiles_g = (a.ntiles - (j0 + g * per_mb) + 2 * per_mb - 1) / (2 * per_mb);
    const int n_chunks = n_tiles_g > 0 ? n_tiles_g * kWChunks : 0;
    auto col_of = [&](int n) { return (j0 + g * per_mb + (n / kWChunks) * 2 * per_mb) * kWN + (n % kWChunks) * 64; };
    auto issue = [&](int n) {                      // copy chunk n of the warp's rows into stage n % 2
      if (n < n_chunks) {
        const int c0 = col_of(n) + gq * 8;
        uint8_t* st = wstage + size_t(n % kRowsUStages) * kWStageU;
        if (c0 < a.V) {
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            const int jr = 4 * m + (lane >> 3);
            if (vld[m]) cp_async16(st + jr * kTcRowBytes + ((gq ^ (jr & 7)) << 4), a.U + size_t(rks[m]) * a.V + c0);
          }
        }
      }
      cp_async_commit();
    };
    issue(0);
    issue(1);
    int n = 0, i = g;
    for (int t = j0 + g * per_mb; t < a.ntiles; t += 2 * per_mb, i += 2) {
      if (!__all_sync(0xffffffffu, mbar_wait_parity(&bar_tfull[g], (i >> 1) & 1, kTcMaxPolls))) {
        s_err = 1;
        break;
      }
      tc::fence_after_sync();
      for (int c = 0; c < kWChunks; ++c, ++n) {
        float acc0[32], acc1[32];
        const uint32_t taddr = tmem + (uint32_t(qd * 32) << 16) + uint32_t(g * kWN + c * 64);
        tc::tmem_ld32(taddr, acc0);
        tc::tmem_ld32(taddr + 32, acc1);
        tc::tmem_ld_wait();
        if (c == kWChunks - 1) {
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_tempty[g]);
        }
        cp_async_wait_group<1>();                   // this lane's copies of chunk n have landed
        __syncwarp();                               // ... and every other lane's
        uint8_t* st = wstage + size_t(n % kRowsUStages) * kWStageU;
        uint8_t* mine = st + lane * kTcRowBytes;
        uint4 u[8];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) u[cc] = *reinterpret_cast<const uint4*>(mine + ((cc ^ (lane & 7)) << 4));
        const int n0 = t * kWN + c * 64;
        uint4 o[8];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          const uint32_t wv[4] = {u[cc].x, u[cc].y, u[cc].z, u[cc].w};
          uint32_t ow[4];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const int j = 8 * cc + e;
            const float2 ub = make_float2(__uint_as_float(wv[e >> 1] << 16), __uint_as_float(wv[e >> 1] & 0xFFFF0000u));
            const float2 ac = j < 32 ? make_float2(acc0[j], acc0[j + 1]) : make_float2(acc1[j - 32], acc1[j - 31]);
            const float2 x = add2(ub, ac);
            ow[e >> 1] = pack_bf16x2(x.x, x.y);   // the rounding the draws used
          }
          o[cc] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
        }
        __syncwarp();                               // every lane has read its U row
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) *reinterpret_cast<uint4*>(mine + ((cc ^ (lane & 7)) << 4)) = o[cc];
        __syncwarp();                               // the warp's logits are staged
        if (n0 + gq * 8 < a.V) {
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            const int jr = 4 * m + (lane >> 3);
            const uint4 v = *reinterpret_cast<const uint4*>(st + jr * kTcRowBytes + ((gq ^ (jr & 7)) << 4));
            if (vld[m]) *reinterpret_cast<uint4*>(a.out + size_t(rks[m]) * a.V + n0 + gq * 8) = v;
          }
        }
        __syncwarp();                               // the staging is read: refill it
        issue(n + 2);
      }
    }
    cp_async_wait_all();
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kTcEpiWarps + 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kWTmemCols);
  }
  if (threadIdx.x == 0 && s_err) record_device_error(a.workspace, SPECV_ERR_TIMEOUT);
}

namespace {
// Workspace: header | tile partials [R, ceil(V / 64)] | float32 logits [R, V]
// (when the caller keeps none)
struct MarkovLayout {
  size_t part_off, scratch_off, total;
};
MarkovLayout markov_layout(int R, int V, int rank) {
  (void)rank;
  MarkovLayout L;
  size_t off = kHeaderBytes;
  L.part_off = off;
  off = align256(off + size_t(R) * ((V + kTcBN - 1) / kTcBN) * sizeof(MarkovPart));
  L.scratch_off = off;
  off = align256(off + size_t(R) * V * sizeof(float));
  L.total = off;
  return L;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::atomic<void*> fn{nullptr};
  void* p = fn.load(std::memory_order_acquire);
  if (p == nullptr) {
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || p == nullptr)
      return nullptr;
    fn.store(p, std::memory_order_release);
  }
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
}

// W2 [rank, V] bf16 as [64-column x 64-row] 128-byte-swizzled boxes
bool encode_w2(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* m, const void* W2, int rank, int V) {
  const cuuint64_t gdim[2] = {cuuint64_t(V), cuuint64_t(rank)};
  const cuuint64_t gstride[1] = {cuuint64_t(V) * 2};
  const cuuint32_t box[2] = {uint32_t(kTcBN), 64};
  const cuuint32_t es[2] = {1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W2), gdim, gstride, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

constexpr int kPairTN = 256;      // markov_tc2 tile width (128: four accumulators, measured slower)

// Clusters of two CTAs of `fn` (one CTA per SM) that can be resident at once;
// 0 on failure.  Cached per device.
int pair_clusters(const void* fn, size_t smem_bytes) {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kWThreads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n < 1) {
      (void)cudaGetLastError();
      return 0;
    }
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}
}  // namespace

}  // namespace specv

using namespace specv;

extern "C" size_t specv_markov_draft_workspace_size(int R, int gamma, int V, int rank) {
  if (R < 0 || gamma < 0 || V < 1 || rank < 1 || rank > SPECV_MAX_MARKOV_RANK) return 0;
  return markov_layout(R, V, rank).total;
}

extern "C" specv_status specv_markov_draft(const void* U, const void* W1, const void* W2, const int32_t* anchor,
                                           const float* uniforms, int R, int gamma, int V, int rank, float temperature,
                                           int32_t* draft_tokens, void* draft_logits, specv_dtype logits_out_dtype,
                                           void* workspace, size_t workspace_bytes, void* stream) {
  if (R < 0 || gamma < 0 || V < 1 || rank < 1 || rank > SPECV_MAX_MARKOV_RANK || rank % 16 != 0)
    return SPECV_ERR_INVALID_ARG;
  if (!(temperature >= 0.f) || !isfinite(temperature) || (temperature > 0.f && temperature < kMinTemperature))
    return SPECV_ERR_INVALID_ARG;
  if (logits_out_dtype != SPECV_F32 && logits_out_dtype != SPECV_BF16) return SPECV_ERR_INVALID_ARG;
  if (R == 0 || gamma == 0) return SPECV_OK;
  if (!U || !W1 || !W2 || !anchor || !draft_tokens || !workspace) return SPECV_ERR_INVALID_ARG;
  if (temperature > 0.f && !uniforms) return SPECV_ERR_INVALID_ARG;
  if (!aligned_to(U, 2) || !aligned_to(W1, 2) || !aligned_to(W2, 2) || !aligned_to(anchor, 4) ||
      !aligned_to(uniforms, 4) || !aligned_to(draft_tokens, 4) || !aligned_to(workspace, 256) ||
      !aligned_to(draft_logits, logits_out_dtype == SPECV_BF16 ? 2 : 4))
    return SPECV_ERR_INVALID_ARG;
  const MarkovLayout L = markov_layout(R, V, rank);
  if (workspace_bytes < L.total) return SPECV_ERR_INVALID_ARG;
  if ((V + kTcBN - 1) / kTcBN > kSampleThreads * kSampleMaxPer) return SPECV_ERR_UNSUPPORTED;   // V > 262144
  specv_status s = check_device();
  if (s != SPECV_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(workspace);
  MarkovArgs a;
  a.U = static_cast<const uint16_t*>(U);
  a.W1 = static_cast<const uint16_t*>(W1);
  a.W2 = static_cast<const uint16_t*>(W2);
  a.anchor = anchor;
  a.uniforms = uniforms;
  a.tokens = draft_tokens;
  if (draft_logits) {
    a.logits = draft_logits;                    // [R, gamma, V]
    a.logits_bf16 = logits_out_dtype == SPECV_BF16;
    a.lstride_r = long(gamma) * V;
  } else {
    a.logits = base + L.scratch_off;            // [R, V], reused by every step (CUDA-core form)
    a.logits_bf16 = logits_out_dtype == SPECV_BF16;   // the precision the draw uses
    a.lstride_r = V;
  }
  a.part = reinterpret_cast<MarkovPart*>(base + L.part_off);
  a.workspace = workspace;
  a.R = R;
  a.gamma = gamma;
  a.V = V;
  a.rank = rank;
  a.greedy = temperature == 0.f;
  a.c2 = a.greedy ? 0.f : kLog2e / temperature;
  const bool tc_shape = rank % 64 == 0 && rank <= kTcMaxKC * 64 && V % 8 == 0 && aligned_to(U, 16) &&
                        aligned_to(W1, 16) && aligned_to(W2, 16) && (!draft_logits || aligned_to(draft_logits, 16));
  PFN_cuTensorMapEncodeTiled_v12000 encode = tc_shape ? tensor_map_encoder() : nullptr;
  const int nsm = sm_count();
  if (encode != nullptr && nsm > 0) {
    // tensor-core form: per step the GEMM + epilogue and the sampler
    // tensor maps: W2 [rank, V]; U [R, gamma, V]; logits [R, slots, V] (slots = gamma, or 1 for the scratch row)
    const long slots = draft_logits ? gamma : 1;
    const bool lbf = a.logits_bf16 != 0;
    CUtensorMap tmap_w2, tmap_u, tmap_l;
    if (!encode_w2(encode, &tmap_w2, W2, rank, V)) return SPECV_ERR_CUDA;
    {
      const cuuint64_t gdim[3] = {cuuint64_t(V), cuuint64_t(gamma), cuuint64_t(R)};
      const cuuint64_t gstride[2] = {cuuint64_t(V) * 2, cuuint64_t(gamma) * V * 2};
      const cuuint32_t box[3] = {uint32_t(kTcBN), 1, uint32_t(kTcBM)};
      const cuuint32_t es[3] = {1, 1, 1};
      if (encode(&tmap_u, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(U), gdim, gstride, box, es,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return SPECV_ERR_CUDA;
    }
    {
      const cuuint64_t esz = lbf ? 2 : 4;
      const cuuint64_t gdim[3] = {cuuint64_t(V), cuuint64_t(slots), cuuint64_t(R)};
      const cuuint64_t gstride[2] = {cuuint64_t(V) * esz, cuuint64_t(slots) * V * esz};
      const cuuint32_t box[3] = {lbf ? 64u : 32u, 1, 32};
      const cuuint32_t es[3] = {1, 1, 1};
      if (encode(&tmap_l, lbf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.logits,
                 gdim, gstride, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return SPECV_ERR_CUDA;
    }
    // No logits kept and two or more 128-request blocks: CTA pairs (markov_tc2),
    // two blocks per pair.  Otherwise single CTAs: 256-column tiles
    // (markov_tcw), kept bf16 logits leaving through the U slots; kept float32
    // logits (twice the bytes per chunk) use the 64-column kernel, whose own
    // staging lets both halves of a chunk's store go out without waiting.
    const int n_mb = (R + kTcBM - 1) / kTcBM;
    const bool pair = n_mb >= 2 && draft_logits == nullptr;
    const bool wide = draft_logits == nullptr || a.logits_bf16;
    void* tc_fn;
    size_t tc_bytes;
    if (pair) {
      tc_fn = reinterpret_cast<void*>(&markov_tc2_kernel<kPairTN>);
      tc_bytes = kPSmem;
    } else {
      tc_fn = wide ? reinterpret_cast<void*>(&markov_tcw_kernel) : reinterpret_cast<void*>(&markov_tc_kernel<2>);
      tc_bytes = wide ? kWSmem : tc_smem(2, true);
    }
    if (cudaFuncSetAttribute(tc_fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(tc_bytes)) != cudaSuccess)
      return SPECV_ERR_CUDA;
    MarkovTcArgs ta;
    // With no logits kept the epilogue writes only the tile partials and the
    // sampler recomputes the 64 logits of the tile it draws from.
    if (!draft_logits) a.logits = nullptr;
    a.tile_w = kTcBN;
    a.ntile = (V + kTcBN - 1) / kTcBN;
    ta.nkc = rank / 64;
    ta.ntiles = a.ntile;
    dim3 g1;
    if (pair) {
      const int n_pb = (n_mb + 1) / 2;
      const int ncl = pair_clusters(tc_fn, tc_bytes);
      if (ncl < 1) return SPECV_ERR_CUDA;
      ta.per_mb = ncl / n_pb > 0 ? ncl / n_pb : 1;     // clusters per pair of request blocks
      g1 = dim3(unsigned(2 * n_pb * ta.per_mb));
    } else {
      ta.per_mb = nsm / n_mb > 0 ? nsm / n_mb : 1;     // CTAs per request block
      g1 = dim3(unsigned(n_mb * ta.per_mb));
    }
    for (int k = 1; k <= gamma; ++k) {
      a.k = k;
      a.step_off = draft_logits ? long(k - 1) * V : 0;
      ta.m = a;
      ta.lz = draft_logits ? k - 1 : 0;
      // programmatic dependent launch: each grid is scheduled while its
      // predecessor drains and waits (griddepcontrol.wait) for its results
      cudaLaunchAttribute at[2];
      at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      at[0].val.programmaticStreamSerializationAllowed = 1;
      at[1].id = cudaLaunchAttributeClusterDimension;
      at[1].val.clusterDim.x = 2;
      at[1].val.clusterDim.y = 1;
      at[1].val.clusterDim.z = 1;
      cudaLaunchConfig_t cfg = {};
      cfg.stream = st;
      cfg.attrs = at;
      cfg.numAttrs = pair ? 2 : 1;
      void* targs[] = {&tmap_w2, &tmap_u, &tmap_l, &ta};
      void* pargs[] = {&tmap_w2, &tmap_u, &ta};
      cfg.gridDim = g1;
      cfg.blockDim = dim3(pair || wide ? kWThreads : kTcThreads);
      cfg.dynamicSmemBytes = tc_bytes;
      if (cudaLaunchKernelExC(&cfg, tc_fn, pair ? pargs : targs) != cudaSuccess)
        return SPECV_ERR_CUDA;
      cfg.numAttrs = 1;
      void* sargs[] = {&a};
      cfg.gridDim = dim3(unsigned(R));
      cfg.blockDim = dim3(kSampleThreads);
      cfg.dynamicSmemBytes = 0;
      if (cudaLaunchKernelExC(&cfg, reinterpret_cast<void*>(&markov_sample_kernel), sargs) != cudaSuccess)
        return SPECV_ERR_CUDA;
    }
    return SPECV_OK;
  }
  a.tile_w = kMkBN;
  a.ntile = (V + kMkBN - 1) / kMkBN;
  const dim3 g1(unsigned(a.ntile), unsigned((R + kMkBM - 1) / kMkBM));
  for (int k = 1; k <= gamma; ++k) {
    a.k = k;
    a.step_off = draft_logits ? long(k - 1) * V : 0;
    void* args[] = {&a};
    if (cudaLaunchKernel(reinterpret_cast<void*>(&markov_logits_kernel), g1, dim3(kMkThreads), args, 0, st) !=
        cudaSuccess)
      return SPECV_ERR_CUDA;
    if (cudaLaunchKernel(reinterpret_cast<void*>(&markov_sample_kernel), dim3(unsigned(R)), dim3(kSampleThreads), args,
                         0, st) != cudaSuccess)
      return SPECV_ERR_CUDA;
  }
  return SPECV_OK;
}

extern "C" size_t specv_markov_recompute_logits_workspace_size(int R, int gamma) {
  if (R < 0 || gamma < 0 || gamma > SPECV_MAX_GAMMA) return 0;
  return kHeaderBytes + align256(size_t(R) * gamma * sizeof(int32_t));
}

extern "C" specv_status specv_markov_recompute_logits(const void* U, const void* W1, const void* W2,
                                                      const int32_t* anchor, const int32_t* draft_tokens,
                                                      const int32_t* lengths, int R, int gamma, int V, int rank,
                                                      void* draft_logits, void* workspace, size_t workspace_bytes,
                                                      void* stream) {
  if (R < 0 || gamma < 0 || gamma > SPECV_MAX_GAMMA || V < 1 || rank < 1) return SPECV_ERR_INVALID_ARG;
  if (R == 0 || gamma == 0) return SPECV_OK;
  if (!U || !W1 || !W2 || !anchor || !draft_tokens || !draft_logits || !workspace) return SPECV_ERR_INVALID_ARG;
  if (!aligned_to(anchor, 4) || !aligned_to(draft_tokens, 4) || !aligned_to(lengths, 4) ||
      !aligned_to(workspace, 256))
    return SPECV_ERR_INVALID_ARG;
  if (workspace_bytes < specv_markov_recompute_logits_workspace_size(R, gamma)) return SPECV_ERR_INVALID_ARG;
  // the tensor-core tiling of drafting without kept logits, whose sums this reproduces
  if (rank % 64 != 0 || rank > kTcMaxKC * 64 || V % 8 != 0 || !aligned_to(U, 16) || !aligned_to(W1, 16) ||
      !aligned_to(W2, 16) || !aligned_to(draft_logits, 16))
    return SPECV_ERR_UNSUPPORTED;
  specv_status s = check_device();
  if (s != SPECV_OK) return s;
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  const int nsm = sm_count();
  if (encode == nullptr || nsm < 1) return SPECV_ERR_CUDA;
  CUtensorMap tmap_w2;
  if (!encode_w2(encode, &tmap_w2, W2, rank, V)) return SPECV_ERR_CUDA;
  RowsArgs ra;
  ra.U = static_cast<const uint16_t*>(U);
  ra.W1 = static_cast<const uint16_t*>(W1);
  ra.anchor = anchor;
  ra.tokens = draft_tokens;
  ra.lengths = lengths;
  ra.out = static_cast<uint16_t*>(draft_logits);
  ra.rows = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + kHeaderBytes);
  ra.workspace = workspace;
  ra.R = R;
  ra.gamma = gamma;
  ra.V = V;
  ra.rank = rank;
  ra.nkc = rank / 64;
  ra.ntiles = (V + kWN - 1) / kWN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* pargs[] = {&ra};
  if (cudaLaunchKernel(reinterpret_cast<void*>(&markov_rows_prep), dim3(1), dim3(1024), pargs, 0, st) != cudaSuccess)
    return SPECV_ERR_CUDA;
  if (cudaFuncSetAttribute(reinterpret_cast<void*>(&markov_rows_kernel), cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kRowsSmem)) != cudaSuccess)
    return SPECV_ERR_CUDA;
  void* rargs[] = {&tmap_w2, &ra};
  if (launch_dependent(reinterpret_cast<void*>(&markov_rows_kernel), dim3(unsigned(nsm)), dim3(kTcThreads), rargs, st,
                       kRowsSmem) != cudaSuccess)
    return SPECV_ERR_CUDA;
  return SPECV_OK;
}
