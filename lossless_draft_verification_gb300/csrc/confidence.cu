// DSpark's confidence head (sm_103a).
//
// Method (DSpark paper guide, confidence head): for every draft position k a
// light linear projection plus a sigmoid over the backbone hidden state h_k and
// the Markov embedding W1[x_{k-1}] gives c_k, the probability that position k
// passes verification given that every earlier position did:
//   c_{r,k} = sigmoid(w_h . h_{r,k} + w_e . W1[x_{r,k-1}] + b),  x_{r,0} = anchor.
// The scheduler consumes every c_k after the draft is complete, so all
// positions are computed at once, one warp per (request, position): 16-byte
// loads of the bf16 rows of h and W1 (each read once: HBM-bound), eight per lane
// in flight before their FMAs, against the float32 weights, which each CTA
// first copies into shared memory; then a warp sum and the sigmoid.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "host_common.h"

namespace specv {

constexpr int kConfWarps = 8;
constexpr int kConfSmemMaxW = 24 * 1024;    // weights (H + rank floats) staged in shared memory up to this count

struct ConfArgs {
  const uint16_t* h;          // [R, gamma, H] bf16
  const uint16_t* W1;         // [V, rank] bf16
  const float* w;             // [H + rank]
  const int32_t* anchor;      // [R]
  const int32_t* tokens;      // [R, gamma]
  float* conf;                // [R, gamma]
  void* workspace;
  float b;
  int R, gamma, H, V, rank;
  int vec;                    // 16-byte vectors (rows aligned, H and rank multiples of 8)
  int smem_w;                 // vec and H + rank <= kConfSmemMaxW: weights read from shared memory
};

// The same sum with the weights in shared memory: each lane's loads of x for
// eight consecutive steps are issued before their FMAs.  The FMA order per lane
// is the one of dot_bf16 (steps i = lane * 8 + 256 j in increasing j, even
// elements into acc, odd into acc2), so the two give identical results.
// eight bf16 values of x at element i against the staged weights
__device__ __forceinline__ void fma8_sw(uint4 v, const float* sw, int i, float& acc, float& acc2) {
  const float4 w0 = *reinterpret_cast<const float4*>(sw + i);
  const float4 w1 = *reinterpret_cast<const float4*>(sw + i + 4);
  acc = fmaf(__uint_as_float(v.x << 16), w0.x, acc);
  acc2 = fmaf(__uint_as_float(v.x & 0xFFFF0000u), w0.y, acc2);
  acc = fmaf(__uint_as_float(v.y << 16), w0.z, acc);
  acc2 = fmaf(__uint_as_float(v.y & 0xFFFF0000u), w0.w, acc2);
  acc = fmaf(__uint_as_float(v.z << 16), w1.x, acc);
  acc2 = fmaf(__uint_as_float(v.z & 0xFFFF0000u), w1.y, acc2);
  acc = fmaf(__uint_as_float(v.w << 16), w1.z, acc);
  acc2 = fmaf(__uint_as_float(v.w & 0xFFFF0000u), w1.w, acc2);
}

// Steps i = i_start, i_start + 256, ... < n of the lane-strided sum with the
// weights in shared memory, eight loads in flight before their FMAs, continuing
// acc / acc2 (from i_start = lane * 8 the FMA order per lane is dot_bf16's:
// even elements into acc, odd into acc2, so the two give identical results)
__device__ __forceinline__ void dot_bf16_sw(const uint16_t* x, const float* sw, int n, int i_start, float& acc,
                                            float& acc2) {
  for (int i0 = i_start; i0 < n; i0 += 32 * 8 * 8) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * 32 * 8;
      v[u] = i < n ? ldg_stream(x + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * 32 * 8;
      if (i < n) fma8_sw(v[u], sw, i, acc, acc2);
    }
  }
}

// sum_i bf16(x[i]) * w[i] over n elements, lane-strided; float32 FMAs
__device__ __forceinline__ float dot_bf16(const uint16_t* x, const float* w, int n, bool vec, int lane) {
  float acc = 0.f;
  if (vec) {
    // unrolled, two accumulators: each lane keeps several 16-byte loads in flight
    float acc2 = 0.f;
#pragma unroll 8
    for (int i = lane * 8; i < n; i += 32 * 8) {
      const uint4 v = ldg_stream(x + i);
      const float4 w0 = __ldg(reinterpret_cast<const float4*>(w + i));
      const float4 w1 = __ldg(reinterpret_cast<const float4*>(w + i + 4));
      acc = fmaf(__uint_as_float(v.x << 16), w0.x, acc);
      acc2 = fmaf(__uint_as_float(v.x & 0xFFFF0000u), w0.y, acc2);
      acc = fmaf(__uint_as_float(v.y << 16), w0.z, acc);
      acc2 = fmaf(__uint_as_float(v.y & 0xFFFF0000u), w0.w, acc2);
      acc = fmaf(__uint_as_float(v.z << 16), w1.x, acc);
      acc2 = fmaf(__uint_as_float(v.z & 0xFFFF0000u), w1.y, acc2);
      acc = fmaf(__uint_as_float(v.w << 16), w1.z, acc);
      acc2 = fmaf(__uint_as_float(v.w & 0xFFFF0000u), w1.w, acc2);
    }
    acc += acc2;
  } else {
    for (int i = lane; i < n; i += 32) acc = fmaf(__uint_as_float(uint32_t(__ldg(x + i)) << 16), __ldg(w + i), acc);
  }
  return acc;
}

__global__ void __launch_bounds__(kConfWarps * 32) confidence_kernel(ConfArgs a) {
  extern __shared__ __align__(16) float s_w[];   // [H + rank] when smem_w
  if (blockIdx.x == 0 && threadIdx.x == 0) *reinterpret_cast<int*>(a.workspace) = 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (a.smem_w) {
    const int nw = a.H + a.rank;                 // a multiple of 8
    for (int i = threadIdx.x * 4; i < nw; i += kConfWarps * 32 * 4)
      *reinterpret_cast<float4*>(s_w + i) = __ldg(reinterpret_cast<const float4*>(a.w + i));
    __syncthreads();
  }
  const long item = long(blockIdx.x) * kConfWarps + warp;
  if (item >= long(a.R) * a.gamma) return;
  const int r = int(item / a.gamma), k = int(item - long(r) * a.gamma);
  const int x = k == 0 ? __ldg(a.anchor + r) : __ldg(a.tokens + size_t(r) * a.gamma + k - 1);
  const bool bad = x < 0 || x >= a.V;
  float z;
  if (a.smem_w) {
    float acc = 0.f, acc2 = 0.f;
    dot_bf16_sw(a.h + size_t(item) * a.H, s_w, a.H, lane * 8, acc, acc2);
    z = acc + acc2;
    if (!bad) {
      float e = 0.f, e2 = 0.f;
      dot_bf16_sw(a.W1 + size_t(x) * a.rank, s_w + a.H, a.rank, lane * 8, e, e2);
      z += e + e2;
    }
  } else {
    z = dot_bf16(a.h + size_t(item) * a.H, a.w, a.H, a.vec != 0, lane);
    if (!bad) z += dot_bf16(a.W1 + size_t(x) * a.rank, a.w + a.H, a.rank, a.vec != 0, lane);
  }
  z = warp_sum(z);
  if (lane == 0) {
    // sigmoid(z + b) = 1 / (1 + 2^(-(z + b) * log2 e)); saturates to 0 and 1
    const float c = 1.f / (1.f + ex2(-(z + a.b) * kLog2e));
    a.conf[item] = bad ? __int_as_float(0x7fc00000) : c;
    if (bad) record_device_error(a.workspace, SPECV_ERR_DEVICE_DATA);
  }
}

}  // namespace specv

using namespace specv;

extern "C" size_t specv_confidence_head_workspace_size(int R, int gamma) {
  if (R < 0 || gamma < 0) return 0;
  return kHeaderBytes;
}

extern "C" specv_status specv_confidence_head(const void* h, const void* W1, const float* w, float b,
                                              const int32_t* anchor, const int32_t* draft_tokens, int R, int gamma,
                                              int H, int V, int rank, float* conf, void* workspace,
                                              size_t workspace_bytes, void* stream) {
  if (R < 0 || gamma < 0 || H < 0 || V < 1 || rank < 0 || !isfinite(b)) return SPECV_ERR_INVALID_ARG;
  if (R == 0 || gamma == 0) return SPECV_OK;
  if ((H > 0 && !h) || (rank > 0 && !W1) || (H + rank > 0 && !w) || !anchor || (gamma > 1 && !draft_tokens) ||
      !conf || !workspace)
    return SPECV_ERR_INVALID_ARG;
  if (!aligned_to(h, 2) || !aligned_to(W1, 2) || !aligned_to(w, 4) || !aligned_to(anchor, 4) ||
      !aligned_to(draft_tokens, 4) || !aligned_to(conf, 4) || !aligned_to(workspace, 256))
    return SPECV_ERR_INVALID_ARG;
  if (workspace_bytes < kHeaderBytes) return SPECV_ERR_INVALID_ARG;
  specv_status s = check_device();
  if (s != SPECV_OK) return s;
  ConfArgs ca;
  ca.h = static_cast<const uint16_t*>(h);
  ca.W1 = static_cast<const uint16_t*>(W1);
  ca.w = w;
  ca.anchor = anchor;
  ca.tokens = draft_tokens;
  ca.conf = conf;
  ca.workspace = workspace;
  ca.b = b;
  ca.R = R;
  ca.gamma = gamma;
  ca.H = H;
  ca.V = V;
  ca.rank = rank;
  ca.vec = (H % 8 == 0 && rank % 8 == 0 && aligned_to(h, 16) && aligned_to(W1, 16) && aligned_to(w, 16)) ? 1 : 0;
  ca.smem_w = (ca.vec && H + rank <= kConfSmemMaxW) ? 1 : 0;
  const size_t smem = ca.smem_w ? size_t(H + rank) * sizeof(float) : 0;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(reinterpret_cast<const void*>(&confidence_kernel), cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(smem)) != cudaSuccess)
    return SPECV_ERR_CUDA;
  const long items = long(R) * gamma;
  const unsigned grid = unsigned((items + kConfWarps - 1) / kConfWarps);
  void* args[] = {&ca};
  if (cudaLaunchKernel(reinterpret_cast<const void*>(&confidence_kernel), dim3(grid), dim3(kConfWarps * 32), args, smem,
                       static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SPECV_ERR_CUDA;
  return SPECV_OK;
}
