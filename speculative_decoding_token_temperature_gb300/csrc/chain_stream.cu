// Streaming chain verification for 16-byte aligned rows (the common case).
//
// Four kernels chained with programmatic dependent launch; each kernel boundary orders
// one phase's results before the next, so no kernel needs an in-flight fence:
//
//   stats   persistent, one CTA per SM; every warp is an independent pipeline holding
//           three 1-D bulk copies (cp.async.bulk completed on an mbarrier) of its next
//           work items in shared memory.  Item = (row, 4 KB chunk) of logits.  Per chunk:
//           maximum (packed max.NaN.bf16x2 for bf16), then for sampled sequences the sum
//           of 2^((l - m) * log2(e) / T) (packed f32x2 arithmetic, one ex2 per element), or
//           for greedy sequences the lowest index of the maximum.
//   decide  one CTA per sequence: merges every row's chunk summaries in a fixed order,
//           runs the accept tests in order (SD 20.5, "A round of speculative sampling":
//           accept x_i iff u_i * q_i(x_i) < p_i(x_i); J = leading accepts; greedy rows
//           accept iff x_i == argmax, "A round of greedy speculative decoding"), writes the
//           accepted prefix and lists the sequences that draw an extra token.
//   draw    persistent like stats.  Item = (listed sequence, 1024-element chunk) of its
//           drawn row: residual weights (p_J - q_J)+ (q == 0 for the bonus row; SD 20.5,
//           "The speculative sampling rule", "Speculative verification in PyTorch") and
//           their chunk mass.
//   finish  one warp per sequence: locates the chunk whose running mass passes u * S and
//           scans it in index order for the smallest k with C_k > u * S.

#include <climits>

#include "specdec_device.cuh"
#include "specdec_internal.h"

namespace specdec {

namespace {

constexpr uint32_t kNegInfBf16x2 = 0xFF80FF80u;
constexpr float kNaN = __builtin_nanf("");
constexpr int kDecideThreads = 256;
constexpr int kFinishWarps = 8;

__device__ __forceinline__ bool is_greedy(float T) { return !(T >= SPECDEC_GREEDY_TEMPERATURE); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_min(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_max_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ double warp_incl_scan(double v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Merge of (max, normaliser, lowest argmax) summaries of disjoint parts of one row.
struct RowSum {
  float m, Z;
  int z;
};
__device__ __forceinline__ RowSum merge(const RowSum& a, const RowSum& b, float c) {
  RowSum r;
  r.m = max_nan(a.m, b.m);
  const float za = (a.m > -kInf) ? a.Z * ex2((a.m - r.m) * c) : 0.f;
  const float zb = (b.m > -kInf) ? b.Z * ex2((b.m - r.m) * c) : 0.f;
  r.Z = za + zb;
  r.z = min(a.m == r.m ? a.z : INT_MAX, b.m == r.m ? b.z : INT_MAX);
  return r;
}
__device__ __forceinline__ RowSum warp_merge(RowSum s, float c) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    RowSum t;
    t.m = __shfl_xor_sync(0xffffffffu, s.m, o);
    t.Z = __shfl_xor_sync(0xffffffffu, s.Z, o);
    t.z = __shfl_xor_sync(0xffffffffu, s.z, o);
    s = merge(s, t, c);
  }
  return s;
}

template <typename T> struct Vec;  // elements per 16-byte vector
template <> struct Vec<uint16_t> { static constexpr int n = 8; };
template <> struct Vec<float> { static constexpr int n = 4; };

// Bounded-wait failure: record it and wait (bounded) for the copies still in flight to
// this warp's stages before its shared memory can be released.
__device__ __forceinline__ void drain_after_timeout(uint64_t* bar, int stages, uint32_t k, uint32_t issued,
                                                    unsigned* error) {
  atomicOr(error, 1u);
  for (; k < issued; ++k) mbar_wait(&bar[k % stages], (k / stages) & 1u);
}

// ---------------------------------------------------------------------------------
// stats
// ---------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kStatsWarps * 32, 1) chain_stats_stream_kernel(const ChainParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t bars[kStatsWarps][kStatsStages];
  constexpr int VEC = Vec<T>::n;
  constexpr int VPL = kStatsChunkBytes / 16 / 32;  // 16-byte vectors per lane per chunk
  constexpr int EPC = kStatsChunkBytes / static_cast<int>(sizeof(T));  // elements per chunk
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t NW = gridDim.x * kStatsWarps;
  const uint32_t gw = blockIdx.x * kStatsWarps + warp;
  unsigned char* buf = smem + static_cast<size_t>(warp) * kStatsStages * kStatsChunkBytes;
  uint64_t* bar = bars[warp];
  const uint32_t R = P.gamma + 1;
  const uint32_t nch = P.nch;
  const int64_t row_bytes = static_cast<int64_t>(P.V) * sizeof(T);
  const uint32_t n_items = static_cast<uint32_t>(P.B) * R * nch;  // < 2^31 (checked on the host)
  const char* base = static_cast<const char*>(P.logits);

  if (lane == 0) {
    for (int s = 0; s < kStatsStages; ++s) mbar_init(&bar[s], 1);
    mbar_fence_init();
  }
  __syncwarp();

  auto issue = [&](uint32_t it, int s) {
    const uint32_t row = it / nch;
    const int64_t off = static_cast<int64_t>(it - row * nch) * kStatsChunkBytes;
    const uint32_t bytes = static_cast<uint32_t>(min(static_cast<int64_t>(kStatsChunkBytes), row_bytes - off));
    mbar_expect_tx(&bar[s], bytes);
    bulk_copy_g2s(buf + s * kStatsChunkBytes, base + static_cast<int64_t>(row) * row_bytes + off, bytes, &bar[s]);
  };
  uint32_t issued = 0;
  for (uint32_t it = gw; issued < kStatsStages && it < n_items; it += NW, ++issued)
    if (lane == 0) issue(it, issued);

  uint32_t k = 0;
  for (uint32_t it = gw; it < n_items; it += NW, ++k) {
    const int s = static_cast<int>(k % kStatsStages);
    if (!mbar_wait(&bar[s], (k / kStatsStages) & 1u)) {
      if (lane == 0) drain_after_timeout(bar, kStatsStages, k, issued, P.ws.error);
      break;
    }
    const uint32_t row = it / nch;
    const uint32_t ch = it - row * nch;
    const uint32_t b = row / R;
    const int nv = static_cast<int>(min(static_cast<int64_t>(kStatsChunkBytes),
                                        row_bytes - static_cast<int64_t>(ch) * kStatsChunkBytes) / 16);
    const uint4* vb = reinterpret_cast<const uint4*>(buf + s * kStatsChunkBytes);
    uint4 w[VPL];
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int v = lane + 32 * j;
      if (v < nv) {
        w[j] = vb[v];
      } else if constexpr (sizeof(T) == 2) {
        w[j] = make_uint4(kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2);
      } else {
        const uint32_t ni = __float_as_uint(-kInf);
        w[j] = make_uint4(ni, ni, ni, ni);
      }
    }
    __syncwarp();
    // the chunk is in registers: refill this stage with the item kStatsStages steps ahead
    const uint32_t nx = it + kStatsStages * NW;
    const bool refill = nx < n_items && nx > it;
    if (lane == 0 && refill) {
      fence_proxy_async_smem();
      issue(nx, s);
    }
    issued += refill ? 1u : 0u;

    const float Tb = P.greedy_only ? 0.f : __ldg(P.temps + b);
    const bool greedy = P.greedy_only || is_greedy(Tb);
    const float c = greedy ? 0.f : kLog2e / Tb;
    float mt;
    if constexpr (sizeof(T) == 2) {
      uint32_t mm = kNegInfBf16x2;
#pragma unroll
      for (int j = 0; j < VPL; ++j) mm = bf2max(bf2max(mm, w[j].x), bf2max(bf2max(w[j].y, w[j].z), w[j].w));
      mt = max_nan(bf16_lo(mm), bf16_hi(mm));
    } else {
      mt = -kInf;
#pragma unroll
      for (int j = 0; j < VPL; ++j)
        mt = max_nan(mt, max_nan(max_nan(__uint_as_float(w[j].x), __uint_as_float(w[j].y)),
                                 max_nan(__uint_as_float(w[j].z), __uint_as_float(w[j].w))));
    }
    const float m = warp_max(mt);
    float Z = 0.f;
    int z = INT_MAX;
    if (greedy) {
      int idx = INT_MAX;
      if (mt == m) {
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
          const uint32_t ww[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            float v;
            if constexpr (sizeof(T) == 2) v = (e & 1) ? bf16_hi(ww[e >> 1]) : bf16_lo(ww[e >> 1]);
            else v = __uint_as_float(ww[e]);
            if (idx == INT_MAX && v == m && lane + 32 * j < nv)
              idx = static_cast<int>(ch) * EPC + (lane + 32 * j) * VEC + e;
          }
        }
      }
      z = warp_min(idx);
    } else {
      float zt = 0.f;
      if (mt > -kInf) {
        const unsigned long long m2 = f2pack(mt, mt), c2 = f2pack(c, c);
        unsigned long long acc = f2pack(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
          const uint32_t ww[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
          unsigned long long e2[VEC / 2];
#pragma unroll
          for (int p = 0; p < VEC / 2; ++p) {
            unsigned long long x2;
            if constexpr (sizeof(T) == 2) x2 = f2pack(bf16_lo(ww[p]), bf16_hi(ww[p]));
            else x2 = f2pack(__uint_as_float(ww[2 * p]), __uint_as_float(ww[2 * p + 1]));
            float y0, y1;
            f2unpack(f2mul(f2sub(x2, m2), c2), y0, y1);
            e2[p] = f2pack(ex2(y0), ex2(y1));
          }
          unsigned long long vs;
          if constexpr (VEC == 8) vs = f2add(f2add(e2[0], e2[1]), f2add(e2[2], e2[3]));
          else vs = f2add(e2[0], e2[1]);
          acc = f2add(acc, vs);
        }
        float a0, a1;
        f2unpack(acc, a0, a1);
        zt = (a0 + a1) * ex2((mt - m) * c);
      }
      Z = warp_sum(zt);
    }
    if (lane == 0) P.ws.partials[it] = make_float4(m, Z, __int_as_float(z), 0.f);
  }
}

// ---------------------------------------------------------------------------------
// decide: one CTA per sequence
// ---------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kDecideThreads) chain_decide_kernel(const ChainParams P) {
  __shared__ float s_m[kStreamMaxRows], s_Z[kStreamMaxRows];
  __shared__ int s_z[kStreamMaxRows];
  grid_launch_dependents();
  grid_dependency_wait();
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = P.gamma + 1;
  const int nch = P.nch;
  const float Tb = P.greedy_only ? 0.f : __ldg(P.temps + b);
  const bool greedy = P.greedy_only || is_greedy(Tb);
  const float c = greedy ? 0.f : kLog2e / Tb;

  // merge each row's chunk summaries (fixed order: deterministic); warps take rows
  for (int r = warp; r < R; r += kDecideThreads / 32) {
    const float4* pp = P.ws.partials + (static_cast<int64_t>(b) * R + r) * nch;
    RowSum acc;
    acc.m = -kInf;
    acc.Z = 0.f;
    acc.z = INT_MAX;
    for (int q = lane; q < nch; q += 32) {
      const float4 f = __ldcg(pp + q);
      RowSum t;
      t.m = f.x;
      t.Z = f.y;
      t.z = __float_as_int(f.z);
      acc = merge(acc, t, c);
    }
    acc = warp_merge(acc, c);
    if (lane == 0) {
      s_m[r] = acc.m;
      s_Z[r] = acc.Z;
      s_z[r] = acc.z;
    }
  }
  __syncthreads();
  if (warp != 0) return;

  // accept tests, one lane per drafted position
  float m = -kInf, Z = 0.f;
  int z = INT_MAX, st = 0;
  if (lane < R) {
    m = s_m[lane];
    Z = s_Z[lane];
    z = s_z[lane];
    if (!(m == m) || m == kInf) st |= SPECDEC_STATUS_BAD_LOGIT;
    else if (m == -kInf) st |= SPECDEC_STATUS_EMPTY_ROW;
  }
  bool acc = false;
  float px = kNaN;
  int x = -1;
  if (lane < P.gamma) {
    x = __ldg(P.drafts + static_cast<int64_t>(b) * P.gamma + lane);
    if (x < 0 || x >= P.V) {
      st |= SPECDEC_STATUS_BAD_TOKEN;
    } else if (greedy) {
      acc = (x == z);
    } else {
      const T* lrow = static_cast<const T*>(P.logits) + (static_cast<int64_t>(b) * R + lane) * P.V;
      px = ex2((Elem<T>::load(lrow, x) - m) * c) / Z;
      const float qx = __ldg(P.q + (static_cast<int64_t>(b) * P.gamma + lane) * P.V + x);
      if (!(qx >= 0.f && qx < kInf)) {
        st |= SPECDEC_STATUS_BAD_PROB;
      } else if (qx == 0.f) {
        st |= SPECDEC_STATUS_ZERO_Q;
        acc = px > 0.f;
      } else {
        acc = __ldg(P.u + static_cast<int64_t>(b) * R + lane) * qx < px;
      }
    }
    if (P.out_p_draft) P.out_p_draft[static_cast<int64_t>(b) * P.gamma + lane] = px;
  }
  if (!greedy && lane < R) {
    const float uu = __ldg(P.u + static_cast<int64_t>(b) * R + lane);
    if (!(uu >= 0.f && uu < 1.f)) st |= SPECDEC_STATUS_BAD_UNIFORM;
  }
  if (lane == 0 && !P.greedy_only && !(Tb - Tb == 0.f)) st |= SPECDEC_STATUS_BAD_TEMPERATURE;
  st = __reduce_or_sync(0xffffffffu, st);
  const unsigned rej = __ballot_sync(0xffffffffu, !acc) | (0xffffffffu << P.gamma);  // gamma < 32
  int J = __ffs(rej) - 1;
  if (st & SPECDEC_STATUS_ERROR_MASK) J = -1;
  const int src = J < 0 ? 0 : J;
  const int zJ = __shfl_sync(0xffffffffu, z, src);
  const float mJ = __shfl_sync(0xffffffffu, m, src);
  const float ZJ = __shfl_sync(0xffffffffu, Z, src);
  if (lane < R) {
    int tok = -1;
    if (J >= 0) {
      if (lane < J) tok = x;
      else if (lane == J && greedy) tok = zJ;
    }
    P.out_tokens[static_cast<int64_t>(b) * R + lane] = tok;
  }
  if (lane == 0) {
    P.out_J[b] = J;
    if (P.out_status) P.out_status[b] = st;
    const bool draw = (J >= 0) && !greedy;
    SeqState s;
    s.meta = make_int4(J, draw ? 1 : 0, st, 0);
    s.row = make_float4(draw ? mJ : 0.f, draw ? ZJ : 0.f, c,
                        draw ? __ldg(P.u + static_cast<int64_t>(b) * R + P.gamma) : 0.f);
    P.ws.seq[b] = s;
    if (draw) P.ws.draw_list[atomicAdd(P.ws.draw_count, 1u)] = make_int2(b, J);
  }
}

// ---------------------------------------------------------------------------------
// draw
// ---------------------------------------------------------------------------------

// Residual (or target) weights of one 16-byte vector of logits and the matching q values,
// with their fp32 running sum in index order.  Shared by the chunk masses and the final
// scan so both see identical per-vector values.
template <typename T>
__device__ __forceinline__ float vec_weights(const uint4& lw, const float* qv, float mJ, float c,
                                             float invZ, bool no_q, float (&w)[Vec<T>::n],
                                             float& psum, bool& bad_q) {
  constexpr int VEC = Vec<T>::n;
  float l[VEC];
  if constexpr (sizeof(T) == 2) {
    l[0] = bf16_lo(lw.x); l[1] = bf16_hi(lw.x); l[2] = bf16_lo(lw.y); l[3] = bf16_hi(lw.y);
    l[4] = bf16_lo(lw.z); l[5] = bf16_hi(lw.z); l[6] = bf16_lo(lw.w); l[7] = bf16_hi(lw.w);
  } else {
    l[0] = __uint_as_float(lw.x); l[1] = __uint_as_float(lw.y);
    l[2] = __uint_as_float(lw.z); l[3] = __uint_as_float(lw.w);
  }
  const unsigned long long m2 = f2pack(mJ, mJ), c2 = f2pack(c, c), z2 = f2pack(invZ, invZ);
  float acc = 0.f, pacc = 0.f;
#pragma unroll
  for (int p = 0; p < VEC / 2; ++p) {
    float y0, y1;
    f2unpack(f2mul(f2sub(f2pack(l[2 * p], l[2 * p + 1]), m2), c2), y0, y1);
    float p0, p1;
    f2unpack(f2mul(f2pack(ex2(y0), ex2(y1)), z2), p0, p1);
    const float q0 = no_q ? 0.f : qv[2 * p], q1 = no_q ? 0.f : qv[2 * p + 1];
    bad_q |= !(q0 >= 0.f && q0 < kInf) || !(q1 >= 0.f && q1 < kInf);
    w[2 * p] = fmaxf(p0 - q0, 0.f);
    w[2 * p + 1] = fmaxf(p1 - q1, 0.f);
    acc += w[2 * p];
    acc += w[2 * p + 1];
    pacc += p0;
    pacc += p1;
  }
  psum = pacc;
  return acc;
}

template <typename T>
__global__ void __launch_bounds__(kDrawWarps * 32, 1) chain_draw_stream_kernel(const ChainParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t bars[kDrawWarps][kDrawStages];
  constexpr int VEC = Vec<T>::n;
  constexpr int LBYTES = kDrawChunk * static_cast<int>(sizeof(T));
  constexpr int STAGE = LBYTES + kDrawChunk * 4;
  constexpr int VPL = (kDrawChunk / VEC) / 32;
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t NW = gridDim.x * kDrawWarps;
  const uint32_t gw = blockIdx.x * kDrawWarps + warp;
  unsigned char* buf = smem + static_cast<size_t>(warp) * kDrawStages * STAGE;
  uint64_t* bar = bars[warp];
  const int R = P.gamma + 1;
  const uint32_t nchd = P.nchd;

  if (lane == 0) {
    for (int s = 0; s < kDrawStages; ++s) mbar_init(&bar[s], 1);
    mbar_fence_init();
  }
  __syncwarp();
  grid_dependency_wait();  // the decision kernel's list and states are visible from here
  const uint32_t n_items = __ldcg(P.ws.draw_count) * nchd;

  auto issue = [&](uint32_t it, int s) {
    const int2 e = __ldcg(P.ws.draw_list + it / nchd);
    const uint32_t cd = it % nchd;
    const int n = min(kDrawChunk, P.V - static_cast<int>(cd) * kDrawChunk);
    const uint32_t lb = static_cast<uint32_t>(n) * sizeof(T);
    const uint32_t qb = (e.y < P.gamma) ? static_cast<uint32_t>(n) * 4u : 0u;
    mbar_expect_tx(&bar[s], lb + qb);
    const T* src = static_cast<const T*>(P.logits) + (static_cast<int64_t>(e.x) * R + e.y) * P.V +
                   static_cast<int64_t>(cd) * kDrawChunk;
    bulk_copy_g2s(buf + s * STAGE, src, lb, &bar[s]);
    if (qb) {
      const float* qs = P.q + (static_cast<int64_t>(e.x) * P.gamma + e.y) * P.V + static_cast<int64_t>(cd) * kDrawChunk;
      bulk_copy_g2s(buf + s * STAGE + LBYTES, qs, qb, &bar[s]);
    }
  };
  uint32_t issued = 0;
  for (uint32_t it = gw; issued < kDrawStages && it < n_items; it += NW, ++issued)
    if (lane == 0) issue(it, issued);

  uint32_t k = 0;
  for (uint32_t it = gw; it < n_items; it += NW, ++k) {
    const int s = static_cast<int>(k % kDrawStages);
    if (!mbar_wait(&bar[s], (k / kDrawStages) & 1u)) {
      if (lane == 0) drain_after_timeout(bar, kDrawStages, k, issued, P.ws.error);
      break;
    }
    const int2 e = __ldcg(P.ws.draw_list + it / nchd);
    const uint32_t cd = it % nchd;
    const float4 row = __ldcg(&P.ws.seq[e.x].row);
    const bool has_q = e.y < P.gamma;
    const int n = min(kDrawChunk, P.V - static_cast<int>(cd) * kDrawChunk);
    const int nv = n / VEC;
    const float c = row.z, mJ = row.x, invZ = 1.f / row.y;
    const unsigned char* sb = buf + s * STAGE;
    uint4 lw[VPL];
    float qv[VPL][VEC];
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int v = lane + 32 * j;
      if (v < nv) {
        lw[j] = reinterpret_cast<const uint4*>(sb)[v];
        if (has_q) {
#pragma unroll
          for (int q4 = 0; q4 < VEC; q4 += 4) {
            const float4 f = reinterpret_cast<const float4*>(sb + LBYTES)[(v * VEC + q4) / 4];
            qv[j][q4] = f.x; qv[j][q4 + 1] = f.y; qv[j][q4 + 2] = f.z; qv[j][q4 + 3] = f.w;
          }
        }
      }
    }
    __syncwarp();
    const uint32_t nx = it + kDrawStages * NW;
    const bool refill = nx < n_items && nx > it;
    if (lane == 0 && refill) {
      fence_proxy_async_smem();
      issue(nx, s);
    }
    issued += refill ? 1u : 0u;
    float sr = 0.f, sp = 0.f;
    bool bad = false;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int v = lane + 32 * j;
      if (v < nv) {
        float w[VEC], ps;
        sr += vec_weights<T>(lw[j], qv[j], mJ, c, invZ, !has_q, w, ps, bad);
        sp += ps;
      }
    }
    if (__any_sync(0xffffffffu, bad)) sr = kNaN;
    sr = warp_sum(sr);
    sp = warp_sum(sp);
    if (lane == 0) P.ws.draw_mass[static_cast<int64_t>(e.x) * nchd + cd] = make_float2(sr, sp);
  }
}

// ---------------------------------------------------------------------------------
// finish: one warp per sequence
// ---------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kFinishWarps * 32) chain_finish_kernel(const ChainParams P) {
  constexpr int VEC = Vec<T>::n;
  constexpr int VPL = (kDrawChunk / VEC) / 32;  // contiguous vectors per lane in the scan
  grid_launch_dependents();
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * kFinishWarps + (threadIdx.x >> 5);
  if (b >= P.B) return;
  SeqState st;
  st.meta = __ldcg(&P.ws.seq[b].meta);
  if (st.meta.y == 0) return;
  st.row = __ldcg(&P.ws.seq[b].row);
  const int R = P.gamma + 1;
  const int J = st.meta.x;
  const int nchd = P.nchd;
  const float2* dm = P.ws.draw_mass + static_cast<int64_t>(b) * nchd;
  int32_t* tok_out = P.out_tokens + static_cast<int64_t>(b) * R;

  double S = 0.0, Sp = 0.0;
  for (int q = lane; q < nchd; q += 32) {
    const float2 d = __ldcg(dm + q);
    S += static_cast<double>(d.x);
    Sp += static_cast<double>(d.y);
  }
  S = warp_sum(S);
  Sp = warp_sum(Sp);
  if (S != S) {  // a NaN, infinite or negative draft probability in the drawn row
    if (lane < R) tok_out[lane] = -1;
    if (lane == 0) {
      P.out_J[b] = -1;
      if (P.out_status) P.out_status[b] = st.meta.z | SPECDEC_STATUS_BAD_PROB;
    }
    return;
  }
  const bool use_p = !(S > 0.0);  // zero residual after rounding: draw from p
  const double target = static_cast<double>(st.row.w) * (use_p ? Sp : S);

  // the chunk whose running mass first exceeds target (fp64 prefix in chunk order)
  double base = 0.0, base_last = 0.0;
  int cstar = -1, clast = -1;
  for (int q0 = 0; q0 < nchd && cstar < 0; q0 += 32) {
    const int q = q0 + lane;
    double wq = 0.0;
    if (q < nchd) {
      const float2 d = __ldcg(dm + q);
      wq = static_cast<double>(use_p ? d.y : d.x);
    }
    const double incl = warp_incl_scan(wq, lane);
    const double tot = __shfl_sync(0xffffffffu, incl, 31);
    const unsigned pos = __ballot_sync(0xffffffffu, wq > 0.0);
    if (pos) {
      const int hl = 31 - __clz(pos);
      clast = q0 + hl;
      base_last = base + __shfl_sync(0xffffffffu, incl - wq, hl);
    }
    const unsigned hit = __ballot_sync(0xffffffffu, base + incl > target);
    if (hit) {
      const int fl = __ffs(hit) - 1;
      cstar = q0 + fl;
      base = base + __shfl_sync(0xffffffffu, incl - wq, fl);
    } else {
      base += tot;
    }
  }
  if (cstar < 0) {
    cstar = clast < 0 ? 0 : clast;
    base = base_last;
  }

  // scan that chunk in index order: lane l owns VPL contiguous vectors
  const T* lrow = static_cast<const T*>(P.logits) + (static_cast<int64_t>(b) * R + J) * P.V;
  const float* qrow = (J < P.gamma) ? P.q + (static_cast<int64_t>(b) * P.gamma + J) * P.V : nullptr;
  const bool no_q = use_p || qrow == nullptr;
  const float c = st.row.z, mJ = st.row.x, invZ = 1.f / st.row.y;
  const int k0 = cstar * kDrawChunk;
  const int nv = min(kDrawChunk, P.V - k0) / VEC;
  float vsum[VPL];
  double mine = 0.0;
  int last_pos = -1;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int v = lane * VPL + j;
    vsum[j] = 0.f;
    if (v < nv) {
      const uint4 lw = __ldg(reinterpret_cast<const uint4*>(lrow + k0 + v * VEC));
      float qv[VEC];
      if (!no_q) load_q<VEC>(qrow, k0 + v * VEC, qv);
      float w[VEC], ps;
      bool bad = false;
      vsum[j] = vec_weights<T>(lw, qv, mJ, c, invZ, no_q, w, ps, bad);
#pragma unroll
      for (int e = 0; e < VEC; ++e)
        if (w[e] > 0.f) last_pos = k0 + v * VEC + e;
      mine += static_cast<double>(vsum[j]);
    }
  }
  const double incl = warp_incl_scan(mine, lane);
  const unsigned hit = __ballot_sync(0xffffffffu, base + incl > target);
  int y = -1;
  if (hit) {
    const int fl = __ffs(hit) - 1;
    if (lane == fl) {
      double pre = base + (incl - mine);
      for (int j = 0; j < VPL && y < 0; ++j) {
        const int v = lane * VPL + j;
        if (v >= nv) break;
        if (pre + static_cast<double>(vsum[j]) > target) {
          const uint4 lw = __ldg(reinterpret_cast<const uint4*>(lrow + k0 + v * VEC));
          float qv[VEC];
          if (!no_q) load_q<VEC>(qrow, k0 + v * VEC, qv);
          float w[VEC], ps;
          bool bad = false;
          vec_weights<T>(lw, qv, mJ, c, invZ, no_q, w, ps, bad);
          float run = 0.f;
          int lastp = -1;
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            run += w[e];
            if (w[e] > 0.f) lastp = k0 + v * VEC + e;
            if (y < 0 && pre + static_cast<double>(run) > target) y = k0 + v * VEC + e;
          }
          if (y < 0) y = lastp;
        }
        pre += static_cast<double>(vsum[j]);
      }
    }
    y = __shfl_sync(0xffffffffu, y, fl);
  }
  if (y < 0) y = warp_max_int(last_pos);  // rounding put u * S at or past the end
  if (lane == 0) {
    tok_out[J] = y;
    if (use_p && P.out_status) P.out_status[b] = st.meta.z | SPECDEC_STATUS_ZERO_RESIDUAL;
  }
}

// Raise a kernel's dynamic shared-memory limit once per device; `configured` must be a
// flag set private to that kernel.
cudaError_t set_smem(const void* kernel, int bytes, unsigned long long& configured) {
  int dev = 0;
  cudaGetDevice(&dev);
  const unsigned long long bit = 1ull << (dev & 63);
  if (configured & bit) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) configured |= bit;
  return e;
}

template <typename T>
cudaError_t launch_stats_t(const ChainParams& P, cudaStream_t stream) {
  constexpr int smem = kStatsWarps * kStatsStages * kStatsChunkBytes;
  static unsigned long long configured = 0;
  cudaError_t e = set_smem(reinterpret_cast<const void*>(chain_stats_stream_kernel<T>), smem, configured);
  if (e != cudaSuccess) return e;
  return launch_kernel(chain_stats_stream_kernel<T>, dim3(P.grid_stats), dim3(kStatsWarps * 32), smem,
                       stream, 0, P);
}

template <typename T>
cudaError_t launch_draw_t(const ChainParams& P, cudaStream_t stream) {
  constexpr int smem = kDrawWarps * kDrawStages * (kDrawChunk * static_cast<int>(sizeof(T)) + kDrawChunk * 4);
  static unsigned long long configured = 0;
  cudaError_t e = set_smem(reinterpret_cast<const void*>(chain_draw_stream_kernel<T>), smem, configured);
  if (e != cudaSuccess) return e;
  return launch_kernel(chain_draw_stream_kernel<T>, dim3(P.grid_draw), dim3(kDrawWarps * 32), smem, stream, 1, P);
}

}  // namespace

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

cudaError_t launch_chain_stream_stats(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream) {
  return ldt == SPECDEC_BF16 ? launch_stats_t<uint16_t>(P, stream) : launch_stats_t<float>(P, stream);
}

cudaError_t launch_chain_stream_decide(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream) {
  if (ldt == SPECDEC_BF16)
    return launch_kernel(chain_decide_kernel<uint16_t>, dim3(P.B), dim3(kDecideThreads), 0, stream, 1, P);
  return launch_kernel(chain_decide_kernel<float>, dim3(P.B), dim3(kDecideThreads), 0, stream, 1, P);
}

cudaError_t launch_chain_stream_draw(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream) {
  return ldt == SPECDEC_BF16 ? launch_draw_t<uint16_t>(P, stream) : launch_draw_t<float>(P, stream);
}

cudaError_t launch_chain_stream_finish(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream) {
  const dim3 grid((P.B + kFinishWarps - 1) / kFinishWarps);
  if (ldt == SPECDEC_BF16)
    return launch_kernel(chain_finish_kernel<uint16_t>, grid, dim3(kFinishWarps * 32), 0, stream, 1, P);
  return launch_kernel(chain_finish_kernel<float>, grid, dim3(kFinishWarps * 32), 0, stream, 1, P);
}

}  // namespace specdec
