// The DSpark Markov draft head (sm_103a).
//
// Method (DSpark paper guide, Markov head): p_k(v | x_0, x_<k) =
// softmax(U_k(v) + B(x_{k-1}, v)) with the low-rank factorisation B = W1 W2
// (W1 [V, r] used as a row lookup, W2 [r, V] as a logit projection), sampled
// position by position from the anchor x_0.
//
// Per step k (x_{k-1} -> x_k):
//   markov_logits   L = U_k + W1[x_{k-1}] . W2 for a [BM x BN] output tile,
//                   float32 accumulation; the epilogue writes L (float32 or
//                   bf16) and the tile's softmax partials (max * c2,
//                   sum 2^(L*c2 - max*c2)) or, at T = 0, (max, argmax).
//   markov_sample   one warp per request: combines the tile partials, picks the
//                   tile holding u * Z and rescans its BN logits (inverse CDF
//                   over ascending ids), or takes the argmax at T = 0.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "host_common.h"

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
  void* logits;               // output logits base: [R, lstride_r] rows of V (f32 or bf16)
  int logits_bf16;
  long lstride_r;             // elements between consecutive requests in `logits`
  long step_off;              // element offset of this step's row inside a request
  MarkovPart* part;           // [R, ntile]
  void* workspace;
  int R, gamma, V, rank, k;   // k = 1 .. gamma
  int ntile;
  float c2;                   // log2(e)/T, 0 at T = 0
  int greedy;
};

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

__device__ __forceinline__ float round_to_bf16(float x) {
  // round-to-nearest-even to bf16, back to float (finite inputs)
  uint32_t u = __float_as_uint(x);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return __uint_as_float(u & 0xFFFF0000u);
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

__global__ void __launch_bounds__(128) markov_sample_kernel(MarkovArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 4 + warp;
  if (r >= a.R) return;
  const int x_prev = prev_token(a, r);
  const MarkovPart* part = a.part + size_t(r) * a.ntile;
  int tok = -1;
  bool bad = x_prev < 0 || x_prev >= a.V;
  const float u = a.greedy ? 0.f : a.uniforms[size_t(r) * a.gamma + (a.k - 1)];
  if (!a.greedy && !(u >= 0.f && u < 1.f)) bad = true;
  if (!bad && a.greedy) {
    float v = neg_inf();
    int i = 0x7fffffff;
    for (int t = lane; t < a.ntile; t += 32) {
      const MarkovPart p = part[t];
      const int pi = __float_as_int(p.b);
      if (p.a > v || (p.a == v && pi < i)) { v = p.a; i = pi; }
    }
    warp_argmax(v, i);
    tok = i;
  } else if (!bad) {
    float M = neg_inf();
    for (int t = lane; t < a.ntile; t += 32) M = fmaxf(M, part[t].a);
    M = warp_max(M);
    const int per = (a.ntile + 31) / 32;
    const int t0 = lane * per, t1 = min(a.ntile, t0 + per);
    float lsum = 0.f;
    for (int t = t0; t < t1; ++t) lsum += part[t].b * ex2(part[t].a - M);
    const float incl = warp_inclusive_scan(lsum);
    const float total = __shfl_sync(0xffffffffu, incl, 31);
    const float target = u * total;
    const unsigned hit = __ballot_sync(0xffffffffu, incl > target && t1 > t0);
    int sel = -1;
    float base = 0.f;
    const int L = hit ? __ffs(hit) - 1 : 31;
    if (lane == L) {
      float run = incl - lsum;
      for (int t = t0; t < t1; ++t) {
        const float m = part[t].b * ex2(part[t].a - M);
        if (hit && run + m > target && m > 0.f) { sel = t; base = run; break; }
        if (!hit && m > 0.f) { sel = t; base = run; }
        run += m;
      }
    }
    sel = __shfl_sync(0xffffffffu, sel, L);
    base = __shfl_sync(0xffffffffu, base, L);
    if (sel < 0) {
      bad = true;
    } else {
      // rescan the selected tile's columns in index order
      const MarkovPart p = part[sel];
      const float s = ex2(p.a - M);
      const size_t rowbase = size_t(r) * a.lstride_r + a.step_off;
      float w[4];
      float ls = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int v = sel * kMkBN + lane * 4 + c;
        float x = neg_inf();
        if (v < a.V) {
          x = a.logits_bf16 ? bf16_to_f32(reinterpret_cast<const uint16_t*>(a.logits)[rowbase + v])
                            : reinterpret_cast<const float*>(a.logits)[rowbase + v];
        }
        w[c] = __fmul_rn(ex2(fmaf(x, a.c2, -p.a)), s);
        ls += w[c];
      }
      const float inc = warp_inclusive_scan(ls);
      float accv = base + (inc - ls);
      int cand = 0x7fffffff, last = -1;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        accv += w[c];
        const int v = sel * kMkBN + lane * 4 + c;
        if (w[c] > 0.f) last = v;
        if (cand == 0x7fffffff && accv > target && w[c] > 0.f) cand = v;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
        last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
      }
      tok = cand != 0x7fffffff ? cand : last;
      if (tok < 0) bad = true;
    }
  }
  if (lane == 0) {
    a.tokens[size_t(r) * a.gamma + (a.k - 1)] = bad ? -1 : tok;
    if (bad) record_device_error(a.workspace, SPECV_ERR_DEVICE_DATA);
  }
}

namespace {
struct MarkovLayout {
  size_t part_off, scratch_off, total;
  int ntile;
};
MarkovLayout markov_layout(int R, int V) {
  MarkovLayout L;
  L.ntile = (V + kMkBN - 1) / kMkBN;
  size_t off = kHeaderBytes;
  L.part_off = off;
  off = align256(off + size_t(R) * L.ntile * sizeof(MarkovPart));
  L.scratch_off = off;
  off = align256(off + size_t(R) * V * sizeof(float));
  L.total = off;
  return L;
}
}  // namespace

}  // namespace specv

using namespace specv;

extern "C" size_t specv_markov_draft_workspace_size(int R, int gamma, int V, int rank) {
  if (R < 0 || gamma < 0 || V < 1 || rank < 1 || rank > SPECV_MAX_MARKOV_RANK) return 0;
  return markov_layout(R, V).total;
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
  const MarkovLayout L = markov_layout(R, V);
  if (workspace_bytes < L.total) return SPECV_ERR_INVALID_ARG;
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
    a.logits = base + L.scratch_off;            // [R, V] float32, reused by every step
    a.logits_bf16 = 0;
    a.lstride_r = V;
  }
  a.part = reinterpret_cast<MarkovPart*>(base + L.part_off);
  a.workspace = workspace;
  a.R = R;
  a.gamma = gamma;
  a.V = V;
  a.rank = rank;
  a.ntile = L.ntile;
  a.greedy = temperature == 0.f;
  a.c2 = a.greedy ? 0.f : kLog2e / temperature;
  const dim3 g1(unsigned(L.ntile), unsigned((R + kMkBM - 1) / kMkBM));
  const dim3 g2(unsigned((R + 3) / 4));
  for (int k = 1; k <= gamma; ++k) {
    a.k = k;
    a.step_off = draft_logits ? long(k - 1) * V : 0;
    void* args[] = {&a};
    if (cudaLaunchKernel(reinterpret_cast<void*>(&markov_logits_kernel), g1, dim3(kMkThreads), args, 0, st) !=
        cudaSuccess)
      return SPECV_ERR_CUDA;
    if (cudaLaunchKernel(reinterpret_cast<void*>(&markov_sample_kernel), g2, dim3(128), args, 0, st) != cudaSuccess)
      return SPECV_ERR_CUDA;
  }
  return SPECV_OK;
}
