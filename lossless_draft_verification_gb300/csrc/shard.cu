// Vocabulary-sharded verification: the host-side combine of per-shard
// partials (no device code).
//
// When a row's V logits are split into contiguous ascending slices, one per
// GPU (the layout of a tensor-parallel LM head), every quantity the chain,
// tree and Markov paths need per row is a combine of per-shard partials:
//   * softmax normalisers: (max, sum of exponentials) pairs merge by
//     log-sum-exp (DART reading notes §2.3: q and p are full-vocabulary
//     softmaxes; the merge is the same identity the kernels use across tiles);
//   * sum_v min(q, p) and sum_v [q - p]_+ are plain sums over shards (c* and
//     the residual mass, DSpark guide analytic acceptance; DART notes eq. (3));
//   * an inverse-CDF draw over ascending token ids first picks the shard
//     whose cumulative mass passes u * total, then draws inside that shard
//     with the remaining target;
//   * a greedy argmax keeps the larger value and, on equal values, the lower
//     token id (speculative-decoding survey §1.3, greedy = argmax).
// The exchange itself (all-gather of the partials) belongs to the caller's
// communication layer; these functions take the gathered partials.
#include <math.h>
#include <stdint.h>

#include "specv.h"

extern "C" specv_status specv_shard_combine_normalisers(const float* part, int shards, int rows, float* out) {
  if (shards < 1 || rows < 0 || (rows > 0 && (!part || !out))) return SPECV_ERR_INVALID_ARG;
  for (int r = 0; r < rows; ++r) {
    double M = -INFINITY;
    for (int s = 0; s < shards; ++s) {
      const float m = part[(size_t(s) * rows + r) * 2];
      const float z = part[(size_t(s) * rows + r) * 2 + 1];
      if (z > 0.f && double(m) > M) M = double(m);
    }
    double Z = 0.0;
    if (M > -INFINITY)
      for (int s = 0; s < shards; ++s) {
        const float m = part[(size_t(s) * rows + r) * 2];
        const float z = part[(size_t(s) * rows + r) * 2 + 1];
        if (z > 0.f) Z += double(z) * exp2(double(m) - M);
      }
    out[size_t(r) * 2] = M > -INFINITY ? float(M) : -INFINITY;
    out[size_t(r) * 2 + 1] = float(Z);
  }
  return SPECV_OK;
}

extern "C" specv_status specv_shard_pick(const double* mass, int shards, int rows, const float* u,
                                         int32_t* shard_out, double* target_out) {
  if (shards < 1 || rows < 0 || (rows > 0 && (!mass || !u || !shard_out || !target_out)))
    return SPECV_ERR_INVALID_ARG;
  for (int r = 0; r < rows; ++r) {
    double total = 0.0;
    for (int s = 0; s < shards; ++s) {
      const double m = mass[size_t(s) * rows + r];
      if (!(m >= 0.0) || !isfinite(m)) return SPECV_ERR_INVALID_ARG;
      total += m;
    }
    const double ur = double(u[r]);
    if (!(ur >= 0.0 && ur < 1.0)) return SPECV_ERR_INVALID_ARG;
    int pick = -1, last = -1;
    double before = 0.0, before_last = 0.0;
    const double target = ur * total;
    double run = 0.0;
    for (int s = 0; s < shards; ++s) {
      const double m = mass[size_t(s) * rows + r];
      if (m > 0.0) {
        last = s;
        before_last = run;
        if (pick < 0 && run + m > target) {
          pick = s;
          before = run;
        }
      }
      run += m;
    }
    if (pick < 0 && last >= 0) {        // rounding at the top: the last shard with mass
      pick = last;
      before = before_last;
    }
    shard_out[r] = pick;
    target_out[r] = pick >= 0 ? fmax(target - before, 0.0) : 0.0;
  }
  return SPECV_OK;
}

extern "C" specv_status specv_shard_argmax_combine(const float* val, const int32_t* idx, int shards, int rows,
                                                   int32_t* out) {
  if (shards < 1 || rows < 0 || (rows > 0 && (!val || !idx || !out))) return SPECV_ERR_INVALID_ARG;
  for (int r = 0; r < rows; ++r) {
    float best = -INFINITY;
    int32_t bi = INT32_MAX;
    for (int s = 0; s < shards; ++s) {
      const float v = val[size_t(s) * rows + r];
      const int32_t i = idx[size_t(s) * rows + r];
      if (v > best || (v == best && i < bi)) {
        best = v;
        bi = i;
      }
    }
    out[r] = bi == INT32_MAX ? -1 : bi;
  }
  return SPECV_OK;
}
