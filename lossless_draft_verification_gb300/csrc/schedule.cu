// DSpark's greedy throughput scheduler (sm_103a), one CTA.
//
// Method (DSpark paper guide, scheduler section): a_{r,j} = prod_{i<=j} c_{r,i};
// every (r, j) enters one pool sorted by a descending; entries are taken from
// the top, each adding 1 to the verify batch B and a_{r,j} to the expected
// accepted count tau; Theta = tau * SPS(B); the loop stops at the first entry
// with Theta <= Theta_best.  Because a_{r,j} does not increase with j, the
// taken entries of each request form a prefix and l_r is their count.
//
// Parallel form: survival products (float64, left to right, one thread per
// request), a sort of (a, index) pairs -- each warp sorts a chunk in registers
// by a bitonic network, then merge-path levels in shared memory join the
// chunks -- then a block-wide
// int64 prefix sum of the fixed-point increments floor(a * 2^48) (exact, so
// identical to any sequential order), Theta_n for every n at once, and a
// block minimum over the first descent.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "host_common.h"

namespace specv {

constexpr int kSchedThreads = 1024;
constexpr double kQuantum = 281474976710656.0;   // 2^48

struct SchedArgs {
  const float* conf;
  const float* conf_stale;    // global mode: confidences that set K (null: conf)
  int global;                 // 0: greedy with the early stop; 1: global search, dynamic top-K
  const double* sps;
  void* workspace;
  int32_t* lengths;
  double* theta_best;
  int R, gamma, B_max, n_pad;
};

// floor(a * 2^48) for 0 <= a <= 1, from the bits of a in integer arithmetic.
// a * 2^48 is exact in float64 (a power-of-two scaling), so this equals the
// truncation of the float64 product.  (Values outside [0, 1] are flagged as
// bad data before their result is used.)
__device__ __forceinline__ long long fixed48(unsigned long long bits) {
  const int e = int((bits >> 52) & 0x7FF);               // biased exponent
  if (e == 0) return 0;                                  // zero or below 2^-1022
  const unsigned long long m = (bits & 0xFFFFFFFFFFFFFull) | (1ull << 52);
  const int sh = 1027 - e;                               // a * 2^48 = m * 2^(e - 1027)
  if (sh >= 64 || sh <= 0) return 0;
  return static_cast<long long>(m >> sh);
}

__device__ __forceinline__ bool pair_less(unsigned long long ka, int ia, unsigned long long kb, int ib) {
  return ka < kb || (ka == kb && ia < ib);
}

// The pool of (key, idx) sorted ascending (a descending, ties by index) for
// one confidence array; key = ~bits(a_{r,j}), idx = r * gamma + j.  Run by
// the whole block; ends with the sorted pool in key / idx.
template <int EPT>
__device__ __forceinline__ void build_pool(const float* conf, int R, int gamma, int n, int n_pad,
                                           unsigned long long* key, int* idx, long long* pre, int* idx2, int* s_bad) {
  const int tid = threadIdx.x;
  // survival products, one request per thread; the confidences are loaded
  // eight at a time before they are used
  for (int r = tid; r < R; r += kSchedThreads) {
    double prod = 1.0;
    for (int j0 = 0; j0 < gamma; j0 += 8) {
      float cj[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) cj[u] = j0 + u < gamma ? __ldg(conf + size_t(r) * gamma + j0 + u) : 1.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u;
        if (j >= gamma) break;
        const float c = cj[u];
        if (!(c >= 0.f && c <= 1.f)) *s_bad = 1;
        prod = __dmul_rn(prod, double(c));
        key[r * gamma + j] = ~static_cast<unsigned long long>(__double_as_longlong(prod));
        idx[r * gamma + j] = r * gamma + j;
      }
    }
  }
  for (int i = n + tid; i < n_pad; i += kSchedThreads) {
    key[i] = ~0ull;
    idx[i] = 0x7fffffff;
  }
  __syncthreads();

  // Sort (key, idx) ascending; the pairs are distinct (idx breaks ties), so
  // there is one sorted order.  First each warp sorts its chunk of 32 * EPT
  // pairs in registers with a bitonic network (lane l holds chunk elements
  // l * EPT .. l * EPT + EPT - 1; partners at distance >= EPT are in another
  // lane and come by shuffle), then the chunks are merged level by level.
  {
    constexpr int CH = 32 * EPT;
    const int lane = tid & 31;
    const int base = (tid >> 5) * CH + lane * EPT;
    unsigned long long k[EPT];
    int ix[EPT];
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      k[e] = key[base + e];
      ix[e] = idx[base + e];
    }
#pragma unroll
    for (int kk = 2; kk <= CH; kk <<= 1) {
#pragma unroll
      for (int j = kk >> 1; j > 0; j >>= 1) {
        if (j >= EPT) {
#pragma unroll
          for (int e = 0; e < EPT; ++e) {
            const int pos = lane * EPT + e;
            const bool up = (pos & kk) == 0, lower = (pos & j) == 0;
            const unsigned long long ok = __shfl_xor_sync(0xffffffffu, k[e], j / EPT);
            const int oi = __shfl_xor_sync(0xffffffffu, ix[e], j / EPT);
            // the lower position of an ascending pair keeps the smaller pair, etc.
            if ((lower == up) == pair_less(ok, oi, k[e], ix[e])) {
              k[e] = ok;
              ix[e] = oi;
            }
          }
        } else {
#pragma unroll
          for (int e = 0; e < EPT; ++e) {
            if (e & j) continue;
            const int f = e | j;
            const bool up = ((lane * EPT + e) & kk) == 0;
            const bool swap = up ? pair_less(k[f], ix[f], k[e], ix[e]) : pair_less(k[e], ix[e], k[f], ix[f]);
            if (swap) {
              const unsigned long long tk = k[e];
              const int ti = ix[e];
              k[e] = k[f];
              ix[e] = ix[f];
              k[f] = tk;
              ix[f] = ti;
            }
          }
        }
      }
    }
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      key[base + e] = k[e];
      idx[base + e] = ix[e];
    }
  }
  __syncthreads();

  // Merge path: each thread writes EPT consecutive outputs, locating its first
  // one (and the first one of a new block) by binary search over the two runs;
  // the second buffer is the prefix array, unused until the sort is done.
  {
    unsigned long long* kin = key;
    int* iin = idx;
    unsigned long long* kout = reinterpret_cast<unsigned long long*>(pre);
    int* iout = idx2;
    for (int len = 32 * EPT; len < n; len <<= 1) {
      const int p0 = tid * EPT;
      int a0 = 0, la = 0, lb = 0, i = 0, j = 0, blk_end = -1;
      for (int p = p0; p < p0 + EPT && p < n; ++p) {
        if (p >= blk_end) {                      // first output of this thread or of a new block
          const int b0 = (p / (2 * len)) * (2 * len);
          a0 = b0;
          la = min(len, n - b0);
          lb = min(len, n - b0 - la);
          blk_end = b0 + la + lb;
          const int d = p - b0;
          int lo = max(0, d - lb), hi = min(d, la);
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            const int jb = a0 + la + d - 1 - mid;
            if (pair_less(kin[a0 + mid], iin[a0 + mid], kin[jb], iin[jb])) lo = mid + 1;
            else hi = mid;
          }
          i = lo;
          j = d - lo;
        }
        const bool take_a = j >= lb || (i < la && pair_less(kin[a0 + i], iin[a0 + i], kin[a0 + la + j], iin[a0 + la + j]));
        const int src = take_a ? a0 + i : a0 + la + j;
        kout[p] = kin[src];
        iout[p] = iin[src];
        if (take_a) ++i; else ++j;
      }
      __syncthreads();
      unsigned long long* tk = kin; kin = kout; kout = tk;
      int* ti = iin; iin = iout; iout = ti;
    }
    if (kin != key) {                            // the sorted order sits in the second buffer
      for (int q = tid; q < n; q += kSchedThreads) {
        key[q] = kin[q];
        idx[q] = iin[q];
      }
      __syncthreads();
    }
  }
}

template <int EPT>
__global__ void __launch_bounds__(kSchedThreads, 1) schedule_kernel(SchedArgs a) {
  constexpr int N_ARR = kSchedThreads * EPT;     // sorted array length (padding sorts last)
  extern __shared__ __align__(16) unsigned char smem[];
  const int n_pad = N_ARR;
  unsigned long long* key = reinterpret_cast<unsigned long long*>(smem);     // ~bits(a): ascending = a descending
  int* idx = reinterpret_cast<int*>(key + n_pad);
  long long* pre = reinterpret_cast<long long*>(idx + n_pad);                // inclusive prefix of aQ (sorted)
  int* ell = reinterpret_cast<int*>(pre + n_pad);                           // [R]
  int* idx2 = ell + a.R;                                                     // merge buffer of idx
  __shared__ long long s_warp[kSchedThreads / 32];
  __shared__ int s_first;
  __shared__ int s_bad;
  __shared__ double s_bestv[kSchedThreads / 32];
  __shared__ int s_bestm[kSchedThreads / 32];

  const int tid = threadIdx.x;
  const int R = a.R, gamma = a.gamma, n = R * gamma;
  if (tid == 0) {
    *reinterpret_cast<int*>(a.workspace) = 0;
    s_first = n + 1;
    s_bad = 0;
  }
  for (int i = tid; i < R; i += kSchedThreads) ell[i] = 0;

  build_pool<EPT>(a.global && a.conf_stale ? a.conf_stale : a.conf, R, gamma, n, n_pad, key, idx, pre, idx2, &s_bad);

  // fixed-point increments and their inclusive prefix (contiguous chunk per thread)
  const int per = (n_pad + kSchedThreads - 1) / kSchedThreads;
  const int b0 = tid * per;
  long long run = 0;
  for (int i = b0; i < b0 + per && i < n_pad; ++i) {
    long long q = 0;
    if (i < n) q = fixed48(~key[i]);
    run += q;
    pre[i] = run;
  }
  // block exclusive scan of the per-thread totals
  const int warp = tid >> 5, lane = tid & 31;
  long long v = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) s_warp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    long long w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long t = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += t;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  const long long offset = (warp > 0 ? s_warp[warp - 1] : 0) + (v - run);
  for (int i = b0; i < b0 + per && i < n_pad; ++i) pre[i] += offset;
  __syncthreads();

  // Theta_m for m entries taken (m = 0 .. n); first m >= 1 that does not rise
  const long long tau0 = static_cast<long long>(R) * static_cast<long long>(kQuantum);
  auto theta = [&](int m) -> double {          // m entries taken, requires R + m <= B_max
    const long long tau = tau0 + (m > 0 ? pre[m - 1] : 0);
    return __dmul_rn(__ll2double_rn(tau), a.sps[R + m - 1]);
  };
  // each Theta_m once, into the sorted keys' space (not needed any more)
  double* th = reinterpret_cast<double*>(key);              // th[m - 1] = Theta_m
  for (int m = 1 + tid; m <= n; m += kSchedThreads) {
    if (R + m <= a.B_max) {
      th[m - 1] = theta(m);
      if (!(a.sps[R + m - 1] > 0.0)) s_bad = 1;
    }
  }
  __syncthreads();
  const double theta0 = theta(0);
  if (!(a.sps[R - 1] > 0.0) && tid == 0) s_bad = 1;
  int taken = 0;
  double theta_taken = 0.0;
  if (!a.global) {
    // early stop: the first m >= 1 whose Theta does not rise (each thread's
    // first stop in its strided m, then one shared atomic per warp)
    int first = n + 1;
    for (int m = 1 + tid; m <= n; m += kSchedThreads) {
      const bool stop = R + m > a.B_max || !(th[m - 1] > (m > 1 ? th[m - 2] : theta0));
      if (stop) {
        first = m;
        break;
      }
    }
    first = int(__reduce_min_sync(0xffffffffu, unsigned(first)));
    if (lane == 0 && first <= n) atomicMin(&s_first, first);
    __syncthreads();
    taken = s_first - 1;
    theta_taken = theta(taken);
  } else {
    // global search: the m in [0, min(n, B_max - R)] with the largest Theta,
    // the smallest such m on equal values
    const int m_lim = min(n, a.B_max - R);
    double bv = tid == 0 ? theta0 : -1.0;
    int bm = tid == 0 ? 0 : 0x7fffffff;
    for (int m = 1 + tid; m <= m_lim; m += kSchedThreads) {
      const double t = th[m - 1];
      if (t > bv || (t == bv && m < bm)) { bv = t; bm = m; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const double ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int om = __shfl_xor_sync(0xffffffffu, bm, o);
      if (ov > bv || (ov == bv && om < bm)) { bv = ov; bm = om; }
    }
    if (lane == 0) {
      s_bestv[warp] = bv;
      s_bestm[warp] = bm;
    }
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kSchedThreads / 32; ++w)
        if (s_bestv[w] > bv || (s_bestv[w] == bv && s_bestm[w] < bm)) { bv = s_bestv[w]; bm = s_bestm[w]; }
      s_first = bm + 1;
      s_bestv[0] = bv;
    }
    __syncthreads();
    taken = s_first - 1;
    theta_taken = s_bestv[0];
    // the entries themselves: the top `taken` of the current pool
    if (a.conf_stale) {
      __syncthreads();
      build_pool<EPT>(a.conf, R, gamma, n, n_pad, key, idx, pre, idx2, &s_bad);
    }
  }
  for (int i = tid; i < taken; i += kSchedThreads) atomicAdd(&ell[idx[i] / gamma], 1);
  __syncthreads();
  const bool bad = s_bad != 0;
  for (int r = tid; r < R; r += kSchedThreads) a.lengths[r] = bad ? -1 : ell[r];
  if (tid == 0) {
    if (a.theta_best) a.theta_best[0] = bad ? __longlong_as_double(0x7ff8000000000000ll) : theta_taken / kQuantum;
    if (bad) record_device_error(a.workspace, SPECV_ERR_DEVICE_DATA);
  }
}

// Confidence-threshold suffix pruning, one thread per request: the prefix
// survival s_{r,i} = prod_{j<=i} c_{r,j} (float64, left to right) and
// l_r = the number of leading positions with s_{r,i} >= threshold.
struct PruneArgs {
  const float* conf;
  void* workspace;
  int32_t* lengths;
  double threshold;
  int R, gamma;
};

__global__ void __launch_bounds__(256) prune_kernel(PruneArgs a) {
  if (blockIdx.x == 0 && threadIdx.x == 0) *reinterpret_cast<int*>(a.workspace) = 0;
  __syncthreads();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= a.R) return;
  double prod = 1.0;
  int ell = 0;
  bool alive = true, bad = false;
  for (int j = 0; j < a.gamma; ++j) {
    const float c = a.conf[size_t(r) * a.gamma + j];
    if (!(c >= 0.f && c <= 1.f)) bad = true;
    prod = __dmul_rn(prod, double(c));
    alive = alive && prod >= a.threshold;
    ell += alive ? 1 : 0;
  }
  a.lengths[r] = bad ? -1 : ell;
  if (bad) record_device_error(a.workspace, SPECV_ERR_DEVICE_DATA);
}

namespace {
int pow2_at_least(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}
size_t sched_smem(int R, int n_pad) {
  return size_t(n_pad) * (sizeof(unsigned long long) + 2 * sizeof(int) + sizeof(long long)) + size_t(R) * sizeof(int);
}
}  // namespace

}  // namespace specv

using namespace specv;

extern "C" size_t specv_schedule_workspace_size(int R, int gamma) {
  if (R < 0 || gamma < 0 || size_t(R) * gamma > SPECV_MAX_SCHED_ENTRIES) return 0;
  return kHeaderBytes;
}

static specv_status schedule_launch(const float* conf, const float* conf_stale, int global, const double* sps,
                                    int R, int gamma, int B_max, int32_t* lengths, double* theta_best,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  if (R < 0 || gamma < 0 || B_max < 1 || size_t(R) * gamma > SPECV_MAX_SCHED_ENTRIES || R > B_max)
    return SPECV_ERR_INVALID_ARG;
  if (R == 0) return SPECV_OK;
  if ((gamma > 0 && !conf) || !sps || !lengths || !workspace) return SPECV_ERR_INVALID_ARG;
  if (!aligned_to(conf, 4) || !aligned_to(conf_stale, 4) || !aligned_to(sps, 8) || !aligned_to(lengths, 4) ||
      !aligned_to(theta_best, 8) || !aligned_to(workspace, 256))
    return SPECV_ERR_INVALID_ARG;
  if (workspace_bytes < kHeaderBytes) return SPECV_ERR_INVALID_ARG;
  specv_status s = check_device();
  if (s != SPECV_OK) return s;
  SchedArgs sa;
  sa.conf = conf;
  sa.conf_stale = (global && gamma > 0 && conf_stale != conf) ? conf_stale : nullptr;
  sa.global = global;
  sa.sps = sps;
  sa.workspace = workspace;
  sa.lengths = lengths;
  sa.theta_best = theta_best;
  sa.R = R;
  sa.gamma = gamma;
  sa.B_max = B_max;
  const int n_pad = pow2_at_least(R * gamma < 2 ? 2 : R * gamma);
  const int ept = n_pad <= 2 * kSchedThreads ? 2 : n_pad <= 4 * kSchedThreads ? 4 : 8;
  sa.n_pad = ept * kSchedThreads;
  const size_t smem = sched_smem(R, sa.n_pad);
  const void* fn = ept == 2 ? reinterpret_cast<const void*>(&schedule_kernel<2>)
                 : ept == 4 ? reinterpret_cast<const void*>(&schedule_kernel<4>)
                            : reinterpret_cast<const void*>(&schedule_kernel<8>);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
    return SPECV_ERR_CUDA;
  void* args[] = {&sa};
  if (cudaLaunchKernel(fn, dim3(1), dim3(kSchedThreads), args, smem, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SPECV_ERR_CUDA;
  return SPECV_OK;
}

extern "C" specv_status specv_schedule(const float* conf, const double* sps, int R, int gamma, int B_max,
                                       int32_t* lengths, double* theta_best, void* workspace, size_t workspace_bytes,
                                       void* stream) {
  return schedule_launch(conf, nullptr, 0, sps, R, gamma, B_max, lengths, theta_best, workspace, workspace_bytes,
                         stream);
}

extern "C" specv_status specv_schedule_global(const float* conf, const float* conf_stale, const double* sps, int R,
                                              int gamma, int B_max, int32_t* lengths, double* theta_best,
                                              void* workspace, size_t workspace_bytes, void* stream) {
  return schedule_launch(conf, conf_stale, 1, sps, R, gamma, B_max, lengths, theta_best, workspace, workspace_bytes,
                         stream);
}

extern "C" specv_status specv_prune_threshold(const float* conf, int R, int gamma, double threshold,
                                              int32_t* lengths, void* workspace, size_t workspace_bytes,
                                              void* stream) {
  if (R < 0 || gamma < 0 || !(threshold == threshold)) return SPECV_ERR_INVALID_ARG;
  if (R == 0) return SPECV_OK;
  if ((gamma > 0 && !conf) || !lengths || !workspace) return SPECV_ERR_INVALID_ARG;
  if (!aligned_to(conf, 4) || !aligned_to(lengths, 4) || !aligned_to(workspace, 256)) return SPECV_ERR_INVALID_ARG;
  if (workspace_bytes < kHeaderBytes) return SPECV_ERR_INVALID_ARG;
  specv_status s = check_device();
  if (s != SPECV_OK) return s;
  PruneArgs pa;
  pa.conf = conf;
  pa.workspace = workspace;
  pa.lengths = lengths;
  pa.threshold = threshold;
  pa.R = R;
  pa.gamma = gamma;
  void* args[] = {&pa};
  if (cudaLaunchKernel(reinterpret_cast<const void*>(&prune_kernel), dim3(unsigned((R + 255) / 256)), dim3(256), args,
                       0, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SPECV_ERR_CUDA;
  return SPECV_OK;
}
