// Greedy verification of a linearised candidate tree (sm_103a).
//
// Method: DART reading notes §2.3 (last paragraph: at temperature 0 the target
// argmax is checked along the candidate paths) and Algorithm 3 steps 9-10
// (ancestors are present; the accepted path and the correction token are
// committed); speculative-decoding survey §2.3 (the tree is linearised and
// verified by one target forward).
//
// Kernels: the row argmax of every node's target row (argmax_tiles, shared with
// the chain verifier: one pass over R x (N+1) x V logits, the only HBM-heavy
// part), then tree_walk with one CTA per request: node i is accepted iff every
// node on its root path carries the argmax of the row above it (each thread
// walks its node's ancestors, at most max_depth steps), and a block reduction
// picks the deepest accepted node (lowest index on ties).
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "host_common.h"

namespace specv {

constexpr int kTreeThreads = 1024;   // one warp per node, 32 nodes per round

struct TreeArgs {
  const int32_t* parents;     // [R, N+1]
  const int32_t* tokens;      // [R, N+1]
  const ArgRec* arg;          // [R*(N+1), stride]
  void* workspace;
  int32_t* path_len;          // [R]
  int32_t* path_nodes;        // [R, max_depth]
  int32_t* out_token;         // [R]
  long V;
  int N1, max_depth, nwt, stride;
};

__global__ void __launch_bounds__(kTreeThreads) tree_walk_kernel(TreeArgs a) {
  __shared__ int s_g[SPECV_MAX_TREE_NODES];
  __shared__ int s_par[SPECV_MAX_TREE_NODES];
  __shared__ int s_tok[SPECV_MAX_TREE_NODES];
  __shared__ int s_best;
  pdl_wait_primary();                      // the argmax tile records are complete
  const int r = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N1 = a.N1;

  for (int i = warp; i < N1; i += kTreeThreads / 32) {
    const int g = combine_argmax(a.arg + size_t(r * N1 + i) * a.stride, a.nwt);
    if (lane == 0) s_g[i] = g;
  }
  int bad = 0;
  for (int i = threadIdx.x; i < N1; i += kTreeThreads) {
    const int p = a.parents[size_t(r) * N1 + i];
    const int t = a.tokens[size_t(r) * N1 + i];
    s_par[i] = p;
    s_tok[i] = t;
    if (i == 0) bad |= p != -1;
    else bad |= !(p >= 0 && p < i) || !(t >= 0 && t < a.V);
  }
  if (threadIdx.x == 0) s_best = 0;             // the root: depth 0, index 0
  bad = __syncthreads_or(bad);
  if (!bad) {
    for (int i = threadIdx.x; i < N1; i += kTreeThreads) {
      int d = 0, j = i;
      bool ok = true;
      while (j != 0 && d <= a.max_depth) {       // parents precede children: j strictly decreases
        const int p = s_par[j];
        ok = ok && s_tok[j] == s_g[p];
        j = p;
        ++d;
      }
      if (d > a.max_depth) bad = 1;
      // deepest first, then lowest index: key = depth * 2^11 + (2047 - i)
      if (ok && !bad) atomicMax(&s_best, (d << 11) | (2047 - i));
    }
  }
  bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) {
    int32_t* nodes = a.path_nodes + size_t(r) * a.max_depth;
    if (bad) {
      a.path_len[r] = -1;
      a.out_token[r] = -1;
      for (int d = 0; d < a.max_depth; ++d) nodes[d] = -1;
      record_device_error(a.workspace, SPECV_ERR_DEVICE_DATA);
    } else {
      const int best = 2047 - (s_best & 2047);
      const int depth = s_best >> 11;
      for (int d = depth; d < a.max_depth; ++d) nodes[d] = -1;
      int j = best;
      for (int d = depth - 1; d >= 0; --d) {
        nodes[d] = j;
        j = s_par[j];
      }
      a.path_len[r] = depth;
      a.out_token[r] = s_g[best];
    }
  }
}

}  // namespace specv

using namespace specv;

namespace {
size_t tree_bytes(int R, int N, const ArgmaxPlan& p) {
  return kHeaderBytes + align256(size_t(R) * (N + 1) * p.stride * sizeof(ArgRec));
}
}  // namespace

extern "C" size_t specv_verify_tree_greedy_workspace_size(int R, int N, int V, specv_dtype dtype) {
  if (R < 0 || N < 0 || N + 1 > SPECV_MAX_TREE_NODES || V < 1 || (dtype != SPECV_F32 && dtype != SPECV_BF16)) return 0;
  size_t need = 0;
  for (int vec = 0; vec < 2; ++vec) {
    ArgmaxPlan p;
    if (vec && V % (dtype == SPECV_BF16 ? 8 : 4) != 0) continue;
    if (argmax_plan(V, dtype, vec != 0, &p)) {
      const size_t n = tree_bytes(R, N, p);
      if (n > need) need = n;
    }
  }
  return need;
}

extern "C" specv_status specv_verify_tree_greedy(const void* target_logits, specv_dtype dtype, const int32_t* parents,
                                                 const int32_t* tokens, int R, int N, int V, int max_depth,
                                                 int32_t* path_len, int32_t* path_nodes, int32_t* out_token,
                                                 void* workspace, size_t workspace_bytes, void* stream) {
  if (dtype != SPECV_F32 && dtype != SPECV_BF16) return SPECV_ERR_INVALID_ARG;
  if (R < 0 || N < 0 || N + 1 > SPECV_MAX_TREE_NODES || V < 1 || max_depth < 1 || max_depth > SPECV_MAX_TREE_DEPTH)
    return SPECV_ERR_INVALID_ARG;
  if (R == 0) return SPECV_OK;
  const size_t esz = dtype == SPECV_BF16 ? 2 : 4;
  if (!target_logits || !parents || !tokens || !path_len || !path_nodes || !out_token || !workspace)
    return SPECV_ERR_INVALID_ARG;
  if (!aligned_to(target_logits, esz) || !aligned_to(parents, 4) || !aligned_to(tokens, 4) ||
      !aligned_to(path_len, 4) || !aligned_to(path_nodes, 4) || !aligned_to(out_token, 4) ||
      !aligned_to(workspace, 256))
    return SPECV_ERR_INVALID_ARG;
  ArgmaxPlan p;
  if (!argmax_plan(V, dtype, rows_16b_ok(target_logits, V, dtype), &p)) return SPECV_ERR_UNSUPPORTED;
  if (workspace_bytes < tree_bytes(R, N, p)) return SPECV_ERR_INVALID_ARG;
  specv_status s = check_device();
  if (s != SPECV_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ArgRec* arg = reinterpret_cast<ArgRec*>(static_cast<char*>(workspace) + kHeaderBytes);
  s = launch_argmax_rows(p, dtype, target_logits, R, N + 1, N + 1, nullptr, 0, 0, V, workspace, arg, true, st);
  if (s != SPECV_OK) return s;
  TreeArgs ta;
  ta.parents = parents;
  ta.tokens = tokens;
  ta.arg = arg;
  ta.workspace = workspace;
  ta.path_len = path_len;
  ta.path_nodes = path_nodes;
  ta.out_token = out_token;
  ta.V = V;
  ta.N1 = N + 1;
  ta.max_depth = max_depth;
  ta.nwt = p.nwt;
  ta.stride = p.stride;
  void* args[] = {&ta};
  if (launch_dependent(reinterpret_cast<void*>(&tree_walk_kernel), dim3(R), dim3(kTreeThreads), args, st) !=
      cudaSuccess)
    return SPECV_ERR_CUDA;
  return SPECV_OK;
}
