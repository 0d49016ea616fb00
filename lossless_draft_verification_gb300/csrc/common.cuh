// Device-side building blocks shared by the verification kernels (sm_103a).
//
// Logit rows are streamed in "warp tiles": a warp owns TILE = 32 * VPT * VW
// consecutive elements of one row, lane l holding the VPT vectors
// (tile_start + (j * 32 + l) * VW), j = 0 .. VPT-1, each of VW elements
// (16 bytes: 8 bf16 or 4 float, or one element on the unaligned path).  Every
// warp-wide load instruction therefore covers 512 contiguous bytes.  Rows are
// kept in registers between the passes of a kernel; the same layout is used
// again when one tile is rescanned for inverse-CDF sampling, so the two passes
// see bit-identical per-element values.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "specv.h"

namespace specv {

constexpr int kWarp = 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kBf16NegInf = 0xFF80u;
constexpr uint32_t kF32NegInfBits = 0xFF800000u;

// ---------------------------------------------------------------------------
// scalar helpers
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float neg_inf() { return __uint_as_float(kF32NegInfBits); }

// maximum over the warp in one instruction (exact; NaN inputs are ignored, as
// by fmaxf)
__device__ __forceinline__ float warp_max(float v) {
  float m;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(m) : "f"(v));
  return m;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// inclusive prefix sum across the warp (lane order)
__device__ __forceinline__ float warp_inclusive_scan(float v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    float t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// (value, index) argmax across the warp: larger value wins, lower index on ties
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, o);
    int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
  }
}

// read-only global loads that bypass L1 allocation (streamed exactly once)
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------
// thread-block cluster primitives (inline PTX)
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// address of `p` (a shared-memory variable of this CTA) in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t cluster_map_shared(const void* p, uint32_t rank) {
  uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  return remote;
}

__device__ __forceinline__ void st_shared_cluster_f4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}

__device__ __forceinline__ float4 ld_shared_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// mbarrier + bulk-copy (TMA engine) primitives, inline PTX
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Wait for the phase with the given parity to complete, giving up after
// `max_iter` polls (each poll itself blocks for a hardware-defined interval).
// Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_parity(uint64_t* bar, uint32_t parity, uint32_t max_iter) {
  const uint32_t a = smem_addr(bar);
  for (uint32_t i = 0; i < max_iter; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done) : "r"(a), "r"(parity) : "memory");
    if (done) return true;
  }
  return false;
}

// arrive on an mbarrier given by its shared::cluster address, in this CTA or
// another CTA of the cluster.  The default CTA-scope release: a cluster-scope
// one would also wait for this thread's outstanding global stores.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

// bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global memory into this CTA's shared memory, completing on `bar`
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(dst_smem)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// per-thread 16-byte asynchronous global -> shared copies (Ampere-style cp.async)
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst_smem)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// this thread's copy groups except the N most recent have landed
template <int N>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }


// programmatic dependent launch
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// packed float32 pairs (sm_100+): two IEEE round-to-nearest operations per
// instruction, through the compiler's builtins so that it allocates the pairs
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// register tiles of logits
//
// Elem = uint16_t (bf16 bits) or float.  VEC selects 16-byte vectors (rows
// 16-byte aligned, V a multiple of VW) or single elements.
template <typename Elem, bool VEC>
struct Lanes {
  static constexpr int VW = VEC ? int(16 / sizeof(Elem)) : 1;
  static constexpr int REGS = VEC ? 4 : 1;
};

template <typename Elem, bool VEC>
struct Slot {
  static constexpr int VW = Lanes<Elem, VEC>::VW;
  uint32_t w[Lanes<Elem, VEC>::REGS];

  // element e as float (exact widening); masked elements read -inf
  __device__ __forceinline__ float get(int e) const {
    if constexpr (VEC) {
      if constexpr (sizeof(Elem) == 2) {
        uint32_t x = w[e >> 1];
        return (e & 1) ? __uint_as_float(x & 0xFFFF0000u) : __uint_as_float(x << 16);
      } else {
        return __uint_as_float(w[e]);
      }
    } else {
      return __uint_as_float(w[0]);
    }
  }

  __device__ __forceinline__ void set_neg_inf() {
    if constexpr (VEC) {
      const uint32_t ninf = sizeof(Elem) == 2 ? (kBf16NegInf | (kBf16NegInf << 16)) : kF32NegInfBits;
      w[0] = w[1] = w[2] = w[3] = ninf;
    } else {
      w[0] = kF32NegInfBits;
    }
  }

  // load elements [idx, idx + VW) of `row` (length V); out-of-row lanes read -inf
  __device__ __forceinline__ void load(const Elem* row, long idx, long V) {
    if constexpr (VEC) {
      if (idx + VW <= V) {
        uint4 v = ldg_stream(row + idx);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
      } else {
        // rows are a multiple of VW long on this path: a slot is fully in or out
        const uint32_t ninf = sizeof(Elem) == 2 ? (kBf16NegInf | (kBf16NegInf << 16)) : kF32NegInfBits;
        w[0] = w[1] = w[2] = w[3] = ninf;
      }
    } else {
      if (idx < V) {
        if constexpr (sizeof(Elem) == 2) w[0] = uint32_t(__ldg(reinterpret_cast<const unsigned short*>(row) + idx)) << 16;
        else w[0] = __float_as_uint(__ldg(reinterpret_cast<const float*>(row) + idx));
      } else {
        w[0] = kF32NegInfBits;
      }
    }
  }

  // element e, unpacked by an opaque instruction: the compiler cannot reuse a
  // conversion from an earlier pass, which would keep the unpacked floats live
  __device__ __forceinline__ float get_fresh(int e) const {
    if constexpr (VEC && sizeof(Elem) == 2) {
      uint32_t r;
      if (e & 1) asm volatile("and.b32 %0, %1, 0xffff0000;" : "=r"(r) : "r"(w[e >> 1]));
      else asm volatile("shl.b32 %0, %1, 16;" : "=r"(r) : "r"(w[e >> 1]));
      return __uint_as_float(r);
    } else {
      return get(e);
    }
  }

  // make the words opaque to the compiler (values unchanged), so that a later
  // pass re-derives its floats from them instead of keeping an earlier pass's
  // unpacked floats alive
  __device__ __forceinline__ void launder() {
#pragma unroll
    for (int i = 0; i < Lanes<Elem, VEC>::REGS; ++i) asm volatile("" : "+r"(w[i]));
  }

  // maximum element (exact)
  __device__ __forceinline__ float vmax() const {
    if constexpr (VEC && sizeof(Elem) == 2) {
      uint32_t m;
      asm("max.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(w[0]), "r"(w[1]));
      uint32_t m2;
      asm("max.bf16x2 %0, %1, %2;" : "=r"(m2) : "r"(w[2]), "r"(w[3]));
      asm("max.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(m), "r"(m2));
      return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
    } else {
      float m = get(0);
#pragma unroll
      for (int e = 1; e < VW; ++e) m = fmaxf(m, get(e));
      return m;
    }
  }
};

// element index (within the row) of element e of lane `lane`'s j-th slot in tile t
template <int VPT, int VW>
__device__ __forceinline__ long slot_index(int tile, int j, int lane) {
  return (long(tile) * (32 * VPT) + j * 32 + lane) * VW;
}

// ---------------------------------------------------------------------------
// workspace layout
//
// [0, 256)   header: int32 device error word at offset 0
// then per-entry buffers, each 256-byte aligned.
constexpr size_t kHeaderBytes = 256;

__host__ __device__ __forceinline__ size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__device__ __forceinline__ void record_device_error(void* workspace, int code) {
  atomicCAS(reinterpret_cast<int*>(workspace), 0, code);
}

// Per-row statistics of a chain row pair (target row, draft row), in the
// ex2 domain: Mc = (max logit) * c2 with c2 = log2(e) / T, Z = sum 2^(x*c2 - Mc).
struct RowStats {
  float Mq_c2, Zq, Mp_c2, Zp;
};

// Per-tile partials: the tile's own max (times c2) for q and p, the tile's
// residual mass sum_v [q(v) - p(v)]_+ and the tile's q mass sum_v q(v).
struct TileStats {
  float mq_c2, mp_c2, resid, qmass;
};

// Scales that turn a tile's local exponentials into probabilities:
// q(v) = 2^(x_q * c2 - mq_c2) * sq, p(v) = 2^(x_p * c2 - mp_c2) * sp.
__device__ __forceinline__ float tile_scale(float m_c2, float M_c2, float Z) {
  return ex2(m_c2 - M_c2) / Z;
}

// (value, index) of a row's maximum, per warp tile
struct ArgRec {
  float v;
  int i;
};

// combine a row's tile records (one warp); lowest index among equal maxima
__device__ __forceinline__ int combine_argmax(const ArgRec* tiles, int nwt) {
  const int lane = threadIdx.x & 31;
  float v = neg_inf();
  int i = 0x7fffffff;
  for (int t = lane; t < nwt; t += 32) {
    const ArgRec ar = tiles[t];
    if (ar.v > v || (ar.v == v && ar.i < i)) { v = ar.v; i = ar.i; }
  }
  warp_argmax(v, i);
  return i;
}

}  // namespace specv
