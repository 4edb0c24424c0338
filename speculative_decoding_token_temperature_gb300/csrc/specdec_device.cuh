// Device-side building blocks shared by the verification kernels (sm_103a).
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "specdec.h"

namespace specdec {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kInf = __builtin_huge_valf();

// ---------------------------------------------------------------------------------
// Scalar helpers (inline PTX for the two instructions the hot loops are built on)
// ---------------------------------------------------------------------------------

// 2^x on the special-function unit (PTX ex2.approx.ftz.f32; results below the normal
// range flush to +0, which only drops terms smaller than 2^-126 of the row maximum).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max that propagates NaN (PTX max.NaN.f32), so one NaN logit poisons the row maximum.
__device__ __forceinline__ float max_nan(float a, float b) {
  float y;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
  return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float load(const float* p, int64_t k) { return __ldg(p + k); }
};
template <> struct Elem<uint16_t> {  // bf16 stored as raw 16-bit words
  static __device__ __forceinline__ float load(const uint16_t* p, int64_t k) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(p + k)) << 16);
  }
};

// A vector of VEC consecutive elements converted to fp32.  VEC == 16 / sizeof(T) uses one
// 16-byte load (the caller guarantees 16-byte alignment); VEC == 1 is the scalar path for
// rows that are not 16-byte aligned.
template <typename T, int VEC> struct VecLoad;

template <> struct VecLoad<uint16_t, 8> {
  static __device__ __forceinline__ void load(const uint16_t* p, int64_t k, float (&v)[8]) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(p + k));
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
  }
};
template <> struct VecLoad<float, 4> {
  static __device__ __forceinline__ void load(const float* p, int64_t k, float (&v)[4]) {
    const float4 w = __ldg(reinterpret_cast<const float4*>(p + k));
    v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
  }
};
template <typename T> struct VecLoad<T, 1> {
  static __device__ __forceinline__ void load(const T* p, int64_t k, float (&v)[1]) {
    v[0] = Elem<T>::load(p, k);
  }
};

// fp32 draft probabilities in groups of VEC (VEC in {1, 4, 8}); 16-byte loads when VEC >= 4.
template <int VEC> __device__ __forceinline__ void load_q(const float* p, int64_t k, float (&v)[VEC]) {
  if constexpr (VEC == 1) {
    v[0] = __ldg(p + k);
  } else {
#pragma unroll
    for (int j = 0; j < VEC; j += 4) {
      const float4 w = __ldg(reinterpret_cast<const float4*>(p + k + j));
      v[j] = w.x; v[j + 1] = w.y; v[j + 2] = w.z; v[j + 3] = w.w;
    }
  }
}

// Row reads from global memory (read-only path) or from the rows staged in shared memory.
template <typename T, int VEC, bool SMEM> struct RowAccess {
  static __device__ __forceinline__ void vec(const T* p, int64_t k, float (&v)[VEC]) {
    if constexpr (!SMEM || VEC == 1) {
      VecLoad<T, VEC>::load(p, k, v);
    } else if constexpr (sizeof(T) == 2) {
      const uint4 w = *reinterpret_cast<const uint4*>(p + k);
      v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
      v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
    } else {
      const float4 w = *reinterpret_cast<const float4*>(p + k);
      v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
    }
  }
  static __device__ __forceinline__ float one(const T* p, int64_t k) {
    if constexpr (!SMEM) return Elem<T>::load(p, k);
    else if constexpr (sizeof(T) == 2) return __uint_as_float(static_cast<uint32_t>(p[k]) << 16);
    else return p[k];
  }
  static __device__ __forceinline__ void qvec(const float* p, int64_t k, float (&v)[VEC]) {
    if constexpr (!SMEM) {
      load_q<VEC>(p, k, v);
    } else {
#pragma unroll
      for (int j = 0; j < VEC; j += 4) {
        const float4 w = *reinterpret_cast<const float4*>(p + k + j);
        v[j] = w.x; v[j + 1] = w.y; v[j + 2] = w.z; v[j + 3] = w.w;
      }
    }
  }
  static __device__ __forceinline__ float qone(const float* p, int64_t k) {
    if constexpr (!SMEM) return __ldg(p + k);
    else return p[k];
  }
};

constexpr int kStageCopy = 32768;  // bytes per bulk copy when staging a row

// Order keys of (value, index): a larger key is a larger value, then a smaller index.
// A NaN anywhere gives the canonical NaN's key, above +inf; all ones marks a copy that
// timed out.  -0 is folded into +0 so that equal values tie on their index.
constexpr unsigned long long kKeyTimeout = ~0ull;
__device__ __forceinline__ unsigned long long order_key(float v, int idx, bool nan) {
  uint32_t u = nan ? 0x7fc00000u : __float_as_uint(v + 0.f);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<unsigned long long>(u) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(idx));
}
__device__ __forceinline__ float key_value(unsigned long long k) {
  const uint32_t o = static_cast<uint32_t>(k >> 32);
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}
__device__ __forceinline__ int key_index(unsigned long long k) {
  return static_cast<int>(~static_cast<uint32_t>(k));
}
__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long k) {  // two redux.sync
  const unsigned hi = __reduce_max_sync(0xffffffffu, static_cast<unsigned>(k >> 32));
  const unsigned lo = __reduce_max_sync(0xffffffffu, static_cast<unsigned>(k >> 32) == hi ? static_cast<unsigned>(k) : 0u);
  return (static_cast<unsigned long long>(hi) << 32) | lo;
}

// ---------------------------------------------------------------------------------
// Block reductions and scans (NT threads, fixed order => deterministic)
// ---------------------------------------------------------------------------------

template <int NT> struct Block {
  static constexpr int kWarps = NT / 32;
  static_assert(NT % 32 == 0 && NT <= 1024, "block size");

  // Max with NaN propagation; result broadcast to all threads.
  static __device__ __forceinline__ float max(float v, float* sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) sh[w] = v;
    __syncthreads();
    float r = sh[0];
#pragma unroll
    for (int i = 1; i < kWarps; ++i) r = max_nan(r, sh[i]);
    return r;
  }

  static __device__ __forceinline__ int min_int(int v, int* sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = ::min(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) sh[w] = v;
    __syncthreads();
    int r = sh[0];
#pragma unroll
    for (int i = 1; i < kWarps; ++i) r = ::min(r, sh[i]);
    return r;
  }

  static __device__ __forceinline__ int or_int(int v, int* sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) sh[w] = v;
    __syncthreads();
    int r = 0;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) r |= sh[i];
    return r;
  }

  static __device__ __forceinline__ float sum(float v, float* sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) sh[w] = v;
    __syncthreads();
    float r = 0.f;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) r += sh[i];
    return r;
  }

  // fp64 sum; the cross-warp step runs in warp 0 only (fp64 is slow on this part), and
  // the result is broadcast through sh[kWarps].  sh holds 2 * kWarps doubles.
  static __device__ __forceinline__ double sum(double v, double* sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return cross_warp_sum(v, sh);
  }
  // Sum of fp32 values: fp32 within each warp, fp64 across warps.
  static __device__ __forceinline__ double sum_f(float v, double* sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return cross_warp_sum(static_cast<double>(v), sh);
  }

  // Inclusive prefix sum in thread order (fp64); also returns the block total.
  static __device__ __forceinline__ double inclusive_scan(double v, double* sh, double& total) {
    const int l = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double n = __shfl_up_sync(0xffffffffu, v, o);
      if (l >= o) v += n;
    }
    return cross_warp_scan(v, sh, total);
  }
  // The same for fp32 values: fp32 within each warp, fp64 across warps.
  static __device__ __forceinline__ double inclusive_scan_f(float v, double* sh, double& total) {
    const int l = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float n = __shfl_up_sync(0xffffffffu, v, o);
      if (l >= o) v += n;
    }
    return cross_warp_scan(static_cast<double>(v), sh, total);
  }

 private:
  // v: this warp's total (every lane).  Warp 0 adds the kWarps totals in a fixed order.
  static __device__ __forceinline__ double cross_warp_sum(double v, double* sh) {
    static_assert(kWarps <= 16, "sh holds 2 * kWarps doubles in 32-entry arrays");
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) sh[w] = v;
    __syncthreads();
    if (w == 0) {
      double x = (l < kWarps) ? sh[l] : 0.0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      if (l == 0) sh[kWarps] = x;
    }
    __syncthreads();
    return sh[kWarps];
  }
  // incl: this thread's inclusive prefix within its warp; the warp total is lane 31's.
  static __device__ __forceinline__ double cross_warp_scan(double incl, double* sh, double& total) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 31) sh[w] = incl;
    __syncthreads();
    if (w == 0) {  // inclusive scan of the warp totals
      double x = (l < kWarps) ? sh[l] : 0.0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double n = __shfl_up_sync(0xffffffffu, x, o);
        if (l >= o) x += n;
      }
      __syncwarp();
      if (l < kWarps) sh[kWarps + l] = x;
    }
    __syncthreads();
    total = sh[2 * kWarps - 1];
    return (w ? sh[kWarps + w - 1] : 0.0) + incl;
  }
};

}  // namespace specdec

namespace specdec {

// ---------------------------------------------------------------------------------
// Packed fp32x2 arithmetic (sm_100+ f32x2 instructions) and packed bf16x2 maximum
// ---------------------------------------------------------------------------------

__device__ __forceinline__ unsigned long long f2pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2unpack(unsigned long long r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long f2sub(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2mul(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2add(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// NaN-propagating maximum of two pairs of bf16 values.
__device__ __forceinline__ unsigned long long f2fma(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint32_t bf2max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// ---------------------------------------------------------------------------------
// Bulk copies global -> shared (cp.async.bulk) completed on an mbarrier
// ---------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
// 1-D bulk copy: dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// 1-D bulk copy with an L2 eviction-priority policy (from l2_policy_*).
__device__ __forceinline__ void bulk_copy_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                   uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
// L2 policies: data read once (evicted first) and data read again soon (kept last).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// One arrival without transaction bytes: completes the phase of a count-1 barrier.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait for the phase with the given parity: gives up (returns false) after about
// one second, so a copy that never lands cannot hang the GPU.
constexpr uint64_t kMaxWaitNs = 1000000000ull;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kMaxWaitNs) return false;
  }
}
// Orders this thread's earlier generic-proxy accesses of shared memory before later
// async-proxy (bulk copy) writes to it.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------------
// Thread-block clusters: distributed shared memory and cluster barriers
// ---------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}
// The shared::cluster address of the same shared-memory location in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}
// 16-byte store into (possibly another CTA's) shared memory that completes 16 bytes of
// transaction count on the mbarrier at `remote_bar` in the same CTA as `remote_addr`.
__device__ __forceinline__ void st_async_16(uint32_t remote_addr, const float4& v, uint32_t remote_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
          remote_addr),
      "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(__float_as_uint(v.z)), "r"(__float_as_uint(v.w)),
      "r"(remote_bar)
      : "memory");
}
// Wait for a phase completed by other CTAs' st.async writes (acquire at cluster scope),
// bounded like mbar_wait.  It polls with the non-blocking test_wait: a thread suspended in
// try_wait was measured to resume several microseconds after such a phase completed, which
// on a chain of dependent exchanges costs more than the polling.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();  // one loop shape for every lane (measured faster)
  for (;;) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (global_timer_ns() - t0 > kMaxWaitNs) return false;
  }
}
// Plain 32-bit loads and stores of (possibly another CTA's) shared memory, addressed by
// cluster_map; ordered with respect to other CTAs by cluster_sync_all().
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// Split cluster barrier without memory ordering: every thread arrives, then waits.  After
// mbarrier initialisation (fence.mbarrier_init by the initialising thread) this makes the
// barriers usable by the other CTAs' bulk copies and st.async.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait;" ::: "memory"); }
// Every thread of every CTA in the cluster.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n barrier.cluster.wait.acquire;" ::: "memory");
}

// Programmatic dependent launch: wait for the preceding grid / allow the next one.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace specdec

namespace specdec {

// Token trees whose children were drawn without replacement: SPECDEC_STATUS_BAD_TREE if
// an earlier node (index below j) has node j's parent and token, else 0 -- from (parent,
// token) pairs staged in shared memory, or from global memory with loads going out eight
// pairs at a time.
__device__ __forceinline__ int sibling_repeats_staged(const int* vp, const int* vt, int j) {
  const int a = vp[j], t = vt[j];
  int bad = 0;
#pragma unroll 8
  for (int i = 0; i < j; ++i) bad |= (vp[i] == a && vt[i] == t) ? 1 : 0;
  return bad ? SPECDEC_STATUS_BAD_TREE : 0;
}
__device__ __forceinline__ int sibling_repeats(const int32_t* parents, const int32_t* toks, int j, int a, int t) {
  int bad = 0, i = 0;
  for (; i + 8 <= j; i += 8) {
    int pa[8], tk[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      pa[e] = __ldg(parents + i + e);
      tk[e] = __ldg(toks + i + e);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) bad |= (pa[e] == a && tk[e] == t) ? 1 : 0;
  }
  for (; i < j; ++i) bad |= (__ldg(parents + i) == a && __ldg(toks + i) == t) ? 1 : 0;
  return bad ? SPECDEC_STATUS_BAD_TREE : 0;
}

// q's mass left at a tree node whose children were drawn without replacement,
// Z = 1 - (q at the children rejected so far), as an unevaluated sum hi + lo of two
// floats: each subtraction is exact (Knuth's two-sum), so Z keeps its accuracy however
// small it gets, with fp32 adds only.
struct MassLeft {
  float hi = 1.f, lo = 0.f;
  __device__ __forceinline__ void sub(float x) {
    const float s = __fsub_rn(hi, x);
    const float bv = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bv)), __fsub_rn(-x, bv));
    const float l = __fadd_rn(lo, err);
    hi = __fadd_rn(s, l);
    lo = __fsub_rn(l, __fsub_rn(hi, s));
  }
  __device__ __forceinline__ float value() const { return __fadd_rn(hi, lo); }
};

// Kernel launch that returns its own error (no reliance on cudaGetLastError, which would
// also report unrelated earlier errors of the calling thread).  pdl != 0 lets the kernel
// start while the previous kernel in the stream finishes (programmatic dependent launch);
// such a kernel must call grid_dependency_wait() before reading that kernel's results.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, int pdl, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace specdec
