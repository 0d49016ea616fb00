// Host-side helpers shared by the entry points.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "specv.h"

namespace specv {

// Temperatures in (0, kMinTemperature) are rejected (T = 0 selects greedy):
// log2(e)/T must stay far from float overflow when multiplied by a logit.
constexpr float kMinTemperature = 1e-6f;

inline bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// SPECV_OK when the current device is an sm_103 part (cached per device).
specv_status check_device();

struct ArgRec;

// Row-argmax over warp tiles (chain.cu): plan for a row length, and launch over
// rows (r, k), k < Pout, of a tensor with P rows per request.  Tile records
// go to out[(r * Pout + k) * stride + tile].
struct ArgmaxPlan {
  int vec, vpt, nwt, stride;
};
bool argmax_plan(long V, specv_dtype dtype, bool vec_ok, ArgmaxPlan* p);
specv_status launch_argmax_rows(const ArgmaxPlan& p, specv_dtype dtype, const void* logits, int R, int P, int Pout,
                                const int32_t* lengths, int lim_off, int gamma, long V, void* ws, ArgRec* out,
                                bool clear_error, cudaStream_t st);
// Launch a kernel that begins with griddepcontrol.wait as a programmatic
// dependent of the previous work on `st`: it is scheduled while its
// predecessor drains.
inline cudaError_t launch_dependent(void* fn, dim3 grid, dim3 block, void** args, cudaStream_t st,
                                    size_t smem = 0) {
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

inline bool rows_16b_ok(const void* p, long V, specv_dtype dtype) {
  const int vw = dtype == SPECV_BF16 ? 8 : 4;
  return p == nullptr || ((reinterpret_cast<uintptr_t>(p) & 15) == 0 && V % vw == 0);
}

}  // namespace specv
