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
#ifndef SPECDEC_DRAW_LIST_CACHE
#define SPECDEC_DRAW_LIST_CACHE 256
#endif
constexpr int kDrawListCache = SPECDEC_DRAW_LIST_CACHE;  // draw-list entries kept in shared memory
constexpr float kNaN = __builtin_nanf("");
constexpr int kDecideThreads = 256;

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
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = P.gamma + 1;
  const int nch = P.nch;
  const float Tb = P.greedy_only ? 0.f : __ldg(P.temps + b);
  const bool greedy = P.greedy_only || is_greedy(Tb);
  const float c = greedy ? 0.f : kLog2e / Tb;

  // Inputs only (drafts, the logit and q at each draft, uniforms): fetched before waiting
  // for the statistics kernel, so these loads overlap its tail.  Lane i < gamma holds
  // position i; lane gamma holds the bonus row and the draw's uniform.
  // Checks of one position, in order: its logits row, then its draft token, then (when
  // sampled) its draft probability and uniform together.
  int x = -1, tok_err = 0, qu_err = 0;
  float lx = 0.f, qx = 0.f, ux = 0.f;
  if (warp == 0) {
    if (lane < P.gamma) {
      x = __ldg(P.drafts + static_cast<int64_t>(b) * P.gamma + lane);
      if (x < 0 || x >= P.V) {
        tok_err = SPECDEC_STATUS_BAD_TOKEN;
      } else if (!greedy) {
        lx = Elem<T>::load(static_cast<const T*>(P.logits) + (static_cast<int64_t>(b) * R + lane) * P.V, x);
        qx = __ldg(P.q + (static_cast<int64_t>(b) * P.gamma + lane) * P.V + x);
        if (!(qx >= 0.f && qx < kInf)) qu_err |= SPECDEC_STATUS_BAD_PROB;
      }
    }
    if (!greedy && lane < R) ux = __ldg(P.u + static_cast<int64_t>(b) * R + lane);
    if (!greedy && lane < P.gamma && !(ux >= 0.f && ux < 1.f)) qu_err |= SPECDEC_STATUS_BAD_UNIFORM;
  }
  grid_dependency_wait();

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

  // Positions are evaluated left to right and evaluation stops at the first rejection
  // (SD 20.5, "A whole round of speculative sampling"); lane i evaluates position i and
  // the first lane that stops -- by an error or a rejection -- decides the round.
  float m = -kInf, Z = 0.f;
  int z = INT_MAX, warn = 0, row_err = 0;
  if (lane < R) {
    m = s_m[lane];
    Z = s_Z[lane];
    z = s_z[lane];
    if (!(m == m) || m == kInf) row_err = SPECDEC_STATUS_BAD_LOGIT;
    else if (m == -kInf) row_err = SPECDEC_STATUS_EMPTY_ROW;
  }
  const int err = row_err ? row_err : (tok_err ? tok_err : qu_err);
  bool acc = false;
  float px = kNaN;
  if (lane < P.gamma && !err) {
    if (greedy) {
      acc = (x == z);
    } else {
      px = ex2((lx - m) * c) / Z;
      if (qx == 0.f) {
        warn |= SPECDEC_STATUS_ZERO_Q;
        acc = px > 0.f;
      } else {
        acc = ux * qx < px;
      }
    }
  }
  const bool stop = (lane < R) && (err != 0 || lane == P.gamma || !acc);
  const int s_stop = __ffs(__ballot_sync(0xffffffffu, stop)) - 1;  // <= gamma
  int st = __shfl_sync(0xffffffffu, err, s_stop);
  st |= __reduce_or_sync(0xffffffffu, lane <= s_stop ? warn : 0);
  if (!P.greedy_only && !(Tb - Tb == 0.f)) st = SPECDEC_STATUS_BAD_TEMPERATURE;
  const float uG = __shfl_sync(0xffffffffu, ux, P.gamma);
  if (!(st & SPECDEC_STATUS_ERROR_MASK) && !greedy && !(uG >= 0.f && uG < 1.f)) st |= SPECDEC_STATUS_BAD_UNIFORM;
  const bool failed = (st & SPECDEC_STATUS_ERROR_MASK) != 0;
  const int J = failed ? -1 : s_stop;
  if (lane < P.gamma && P.out_p_draft)
    P.out_p_draft[static_cast<int64_t>(b) * P.gamma + lane] = (!failed && lane <= J) ? px : kNaN;
  const int zJ = __shfl_sync(0xffffffffu, z, s_stop);
  const float mJ = __shfl_sync(0xffffffffu, m, s_stop);
  const float ZJ = __shfl_sync(0xffffffffu, Z, s_stop);
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
    SeqState sq;
    sq.meta = make_int4(J, draw ? 1 : 0, st, 0);
    sq.row = make_float4(draw ? mJ : 0.f, draw ? ZJ : 0.f, c, draw ? uG : 0.f);
    P.ws.seq[b] = sq;
    if (draw) {
      DrawEntry d;
      d.loc = make_int4(b, J, b, 0);  // (sequence, drawn row, mass slot, 0)
      d.row = make_float4(mJ, c, 1.f / ZJ, 0.f);
      P.ws.draw_list[atomicAdd(P.ws.draw_count, 1u)] = d;
    }
  }
}

// ---------------------------------------------------------------------------------
// draw
// ---------------------------------------------------------------------------------

// Logits of one group of 4 consecutive elements (8 bytes of bf16 or 16 bytes of fp32).
template <typename T> struct Group;
template <> struct Group<uint16_t> {
  using L = uint2;
  static __device__ __forceinline__ void unpack(const L& w, float (&l)[4]) {
    l[0] = bf16_lo(w.x); l[1] = bf16_hi(w.x); l[2] = bf16_lo(w.y); l[3] = bf16_hi(w.y);
  }
};
template <> struct Group<float> {
  using L = uint4;
  static __device__ __forceinline__ void unpack(const L& w, float (&l)[4]) {
    l[0] = __uint_as_float(w.x); l[1] = __uint_as_float(w.y);
    l[2] = __uint_as_float(w.z); l[3] = __uint_as_float(w.w);
  }
};

// Residual (or target) weights of one group of 4 elements and their fp32 running sum in
// index order.  Shared by the chunk masses and the final scan, so both see identical
// per-group values.
// q values are checked by the caller (see q_check): a NaN, an infinity or a negative value
// is reported as SPECDEC_STATUS_BAD_PROB.
template <typename T>
__device__ __forceinline__ float group_weights(const typename Group<T>::L& lw, const float4& q4, float mJ,
                                               float c, float invZ, bool no_q, float (&w)[4]) {
  float l[4];
  Group<T>::unpack(lw, l);
  const float qv[4] = {no_q ? 0.f : q4.x, no_q ? 0.f : q4.y, no_q ? 0.f : q4.z, no_q ? 0.f : q4.w};
  const unsigned long long m2 = f2pack(mJ, mJ), c2 = f2pack(c, c), z2 = f2pack(invZ, invZ);
  float acc = 0.f;
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    float y0, y1;
    f2unpack(f2mul(f2sub(f2pack(l[2 * p], l[2 * p + 1]), m2), c2), y0, y1);
    float p0, p1;
    f2unpack(f2mul(f2pack(ex2(y0), ex2(y1)), z2), p0, p1);
    w[2 * p] = fmaxf(p0 - qv[2 * p], 0.f);
    w[2 * p + 1] = fmaxf(p1 - qv[2 * p + 1], 0.f);
    acc += w[2 * p];
    acc += w[2 * p + 1];
  }
  return acc;
}

// Running check of draft probabilities: the NaN-propagating maximum catches a NaN or an
// infinity, the minimum a negative entry.
struct QCheck {
  float mx = 0.f, mn = 0.f;
  __device__ __forceinline__ void add(const float4& q) {
    mx = max_nan(mx, max_nan(max_nan(q.x, q.y), max_nan(q.z, q.w)));
    mn = fminf(mn, fminf(fminf(q.x, q.y), fminf(q.z, q.w)));
  }
  __device__ __forceinline__ bool bad() const { return !(mx < kInf) || mn < 0.f; }
};

template <typename T>
constexpr int draw_stages() { return sizeof(T) == 2 ? kDrawStages : kDrawStagesF32; }

template <typename T>
constexpr int draw_smem_bytes() {
  return kDrawWarps * draw_stages<T>() * (kDrawChunk * static_cast<int>(sizeof(T)) + kDrawChunk * 4) +
         kDrawListCache * static_cast<int>(sizeof(DrawEntry));
}
static_assert(draw_smem_bytes<uint16_t>() <= 227 * 1024, "bf16 draw stages exceed shared memory");
static_assert(draw_smem_bytes<float>() <= 227 * 1024, "fp32 draw stages exceed shared memory");
static_assert(kStatsWarps * kStatsStages * kStatsChunkBytes <= 227 * 1024, "statistics stages exceed shared memory");

template <typename T>
__global__ void __launch_bounds__(kDrawWarps * 32, 1) chain_draw_stream_kernel(const ChainParams P) {
  constexpr int kStages = draw_stages<T>();
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t bars[kDrawWarps][kStages];
  using GL = typename Group<T>::L;
  constexpr int LBYTES = kDrawChunk * static_cast<int>(sizeof(T));
  constexpr int STAGE = LBYTES + kDrawChunk * 4;
  constexpr int GPL = kDrawChunk / 4 / 32;  // 4-element groups per lane per chunk
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t NW = gridDim.x * kDrawWarps;
  const uint32_t gw = blockIdx.x * kDrawWarps + warp;
  unsigned char* buf = smem + static_cast<size_t>(warp) * kStages * STAGE;
  uint64_t* bar = bars[warp];
  const int R = P.gamma + 1;
  const uint32_t nchd = P.nchd;

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bar[s], 1);
    mbar_fence_init();
  }
  __syncwarp();
  grid_dependency_wait();  // the decision kernel's list is visible from here
  const uint32_t count = __ldcg(P.ws.draw_count);
  const uint32_t n_items = count * nchd;
  // The list, copied to shared memory when it fits: per-item metadata is then a shared
  // load instead of an L2 round trip in every item's critical path.
  DrawEntry* list_s = reinterpret_cast<DrawEntry*>(smem + static_cast<size_t>(kDrawWarps) * kStages * STAGE);
  const bool cached = count <= static_cast<uint32_t>(kDrawListCache);
  if (cached) {
    for (uint32_t i = threadIdx.x; i < count; i += blockDim.x) {
      list_s[i].loc = __ldcg(&P.ws.draw_list[i].loc);
      list_s[i].row = __ldcg(&P.ws.draw_list[i].row);
    }
  }
  __syncthreads();
  const DrawEntry* list = cached ? list_s : P.ws.draw_list;

  auto issue = [&](uint32_t it, int s, int4 loc) {
    const uint32_t cd = it % nchd;
    const int n = min(kDrawChunk, P.V - static_cast<int>(cd) * kDrawChunk);
    const uint32_t lb = static_cast<uint32_t>(n) * sizeof(T);
    const uint32_t qb = (loc.y < P.gamma) ? static_cast<uint32_t>(n) * 4u : 0u;
    mbar_expect_tx(&bar[s], lb + qb);
    const T* src = static_cast<const T*>(P.logits) + (static_cast<int64_t>(loc.x) * R + loc.y) * P.V +
                   static_cast<int64_t>(cd) * kDrawChunk;
    bulk_copy_g2s(buf + s * STAGE, src, lb, &bar[s]);
    if (qb) {
      const float* qs = P.q + (static_cast<int64_t>(loc.x) * P.gamma + loc.y) * P.V + static_cast<int64_t>(cd) * kDrawChunk;
      bulk_copy_g2s(buf + s * STAGE + LBYTES, qs, qb, &bar[s]);
    }
  };
  uint32_t issued = 0;
  for (uint32_t it = gw; issued < kStages && it < n_items; it += NW, ++issued)
    if (lane == 0) issue(it, static_cast<int>(issued), list[it / nchd].loc);

  uint32_t k = 0;
  for (uint32_t it = gw; it < n_items; it += NW, ++k) {
    const int s = static_cast<int>(k % kStages);
    const uint32_t nx = it + kStages * NW;  // the item this stage is refilled with
    const bool refill = nx < n_items && nx > it;
    int4 nloc = make_int4(0, 0, 0, 0);
    if (lane == 0 && refill) nloc = list[nx / nchd].loc;
    DrawEntry cur;
    cur.loc = list[it / nchd].loc;
    cur.row = list[it / nchd].row;
    if (!mbar_wait(&bar[s], (k / kStages) & 1u)) {
      if (lane == 0) drain_after_timeout(bar, kStages, k, issued, P.ws.error);
      break;
    }
    const uint32_t cd = it % nchd;
    const bool has_q = cur.loc.y < P.gamma;
    const int ng = min(kDrawChunk, P.V - static_cast<int>(cd) * kDrawChunk) / 4;
    const unsigned char* sb = buf + s * STAGE;
    GL lw[GPL];
    float4 qv[GPL];
#pragma unroll
    for (int j = 0; j < GPL; ++j) {
      const int g = lane + 32 * j;
      if (g < ng) {
        lw[j] = reinterpret_cast<const GL*>(sb)[g];
        qv[j] = has_q ? reinterpret_cast<const float4*>(sb + LBYTES)[g] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    __syncwarp();
    if (lane == 0 && refill) {
      fence_proxy_async_smem();
      issue(nx, s, nloc);
    }
    issued += refill ? 1u : 0u;
    float sr = 0.f;
    QCheck qc;
#pragma unroll
    for (int j = 0; j < GPL; ++j) {
      if (lane + 32 * j < ng) {
        float w[4];
        sr += group_weights<T>(lw[j], qv[j], cur.row.x, cur.row.y, cur.row.z, !has_q, w);
        qc.add(qv[j]);
      }
    }
    sr = warp_sum(sr);
    if (__any_sync(0xffffffffu, qc.bad())) {
      sr = kNaN;
      if (lane == 0) atomicOr(P.ws.qbad + cur.loc.x, 1);
    }
    if (lane == 0) P.ws.draw_mass[static_cast<int64_t>(cur.loc.z) * nchd + cd] = sr;
  }
}

// ---------------------------------------------------------------------------------
// finish: one warp per sequence
// ---------------------------------------------------------------------------------

// Mass of chunk q of the drawn row: the draw kernel's residual mass, or (zero-residual
// fallback) the mass of p itself, recomputed here.
template <typename T>
__device__ __forceinline__ float chunk_mass(const ChainParams& P, const float* dm, bool use_p, const T* lrow,
                                            int q, float mJ, float c, float invZ) {
  if (!use_p) return __ldcg(dm + q);
  using GL = typename Group<T>::L;
  const int k0 = q * kDrawChunk;
  const int ng = min(kDrawChunk, P.V - k0) / 4;
  float acc = 0.f;
  for (int g = 0; g < ng; ++g) {
    float w[4];
    acc += group_weights<T>(__ldg(reinterpret_cast<const GL*>(lrow + k0) + g), make_float4(0.f, 0.f, 0.f, 0.f),
                            mJ, c, invZ, true, w);
  }
  return acc;
}

// The inverse-CDF draw from one row's chunk masses (one warp): the chunk whose fp64
// running mass first exceeds u * S, then an index-order scan of that chunk for the
// smallest k with C_k > u * S.  invZ scales the weights the masses were made with
// ((p - q)+ with p = 2^((l - m)c) * invZ, q == nullptr for none); a total of zero (possible
// only through rounding) draws from p itself, whose chunk masses are recomputed with
// invZp.  Returns the token, or -1 when a mass is NaN (a bad draft probability).
template <typename T>
__device__ int draw_from_masses(const ChainParams& P, const float* dm, const T* lrow, const float* qrow, float mJ,
                                float c, float invZ, float invZp, float u, int lane, bool& zero_residual) {
  using GL = typename Group<T>::L;
  constexpr int GPL = kDrawChunk / 4 / 32;  // contiguous groups per lane in the scan
  constexpr int CPL = 16;                   // chunk masses per lane kept in registers
  const int nchd = P.nchd;
  zero_residual = false;

  // lane l owns the contiguous chunks [c0, c1); with at most CPL per lane their masses
  // stay in registers
  const int cpl = (nchd + 31) / 32;
  const bool in_regs = cpl <= CPL;
  const int c0 = min(lane * cpl, nchd), c1 = min(c0 + cpl, nchd);
  float wq[CPL];
  double mine = 0.0;
  if (in_regs) {
#pragma unroll
    for (int j = 0; j < CPL; ++j) wq[j] = (c0 + j < c1) ? __ldcg(dm + c0 + j) : 0.f;
#pragma unroll
    for (int j = 0; j < CPL; ++j)
      if (j < c1 - c0) mine += static_cast<double>(wq[j]);
  } else {
    for (int q = c0; q < c1; ++q) mine += static_cast<double>(__ldcg(dm + q));
  }
  double incl = warp_incl_scan(mine, lane);
  double S = __shfl_sync(0xffffffffu, incl, 31);
  if (S != S) return -1;  // a NaN, infinite or negative draft probability in the row
  const bool use_p = !(S > 0.0);  // zero residual after rounding: draw from p instead
  if (use_p) {  // rare: recompute every chunk's mass of p itself (and keep it from here on)
    mine = 0.0;
    if (in_regs) {
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        wq[j] = (j < c1 - c0) ? chunk_mass<T>(P, dm, true, lrow, c0 + j, mJ, c, invZp) : 0.f;
        mine += static_cast<double>(wq[j]);
      }
    } else {
      for (int q = c0; q < c1; ++q) mine += static_cast<double>(chunk_mass<T>(P, dm, true, lrow, q, mJ, c, invZp));
    }
    incl = warp_incl_scan(mine, lane);
    S = __shfl_sync(0xffffffffu, incl, 31);
    zero_residual = true;
  }
  const double target = static_cast<double>(u) * S;

  // Walk this lane's chunks in order: the first whose running mass (from pre) exceeds
  // target, else the last one with mass.  Also returns the running mass before it.
  auto walk = [&](double pre, bool want_cross, int& found, double& before) {
    found = -1;
    before = 0.0;
    int lastpos = -1;
    double prelast = 0.0;
    if (in_regs) {
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        if (j < c1 - c0 && found < 0) {
          const double w = static_cast<double>(wq[j]);
          if (w > 0.0) { lastpos = c0 + j; prelast = pre; }
          if (want_cross && pre + w > target) { found = c0 + j; before = pre; }
          pre += w;
        }
      }
    } else {
      for (int q = c0; q < c1 && found < 0; ++q) {
        const double w = static_cast<double>(chunk_mass<T>(P, dm, use_p, lrow, q, mJ, c, invZp));
        if (w > 0.0) { lastpos = q; prelast = pre; }
        if (want_cross && pre + w > target) { found = q; before = pre; }
        pre += w;
      }
    }
    if (found < 0) { found = lastpos; before = prelast; }
  };

  // the chunk whose running mass first exceeds target (fp64 prefix in chunk order)
  const unsigned hit = __ballot_sync(0xffffffffu, incl > target);
  int cstar = -1;
  double base = 0.0;
  if (hit) {
    const int fl = __ffs(hit) - 1;
    if (lane == fl) walk(incl - mine, true, cstar, base);
    cstar = __shfl_sync(0xffffffffu, cstar, fl);
    base = __shfl_sync(0xffffffffu, base, fl);
  }
  if (cstar < 0) {  // rounding put u * S at or past the end: last chunk with mass
    int lastpos;
    double before;
    walk(incl - mine, false, lastpos, before);
    const int best = warp_max_int(lastpos);
    const unsigned owner = __ballot_sync(0xffffffffu, lastpos == best && best >= 0);
    cstar = best < 0 ? 0 : best;
    base = owner ? __shfl_sync(0xffffffffu, before, __ffs(owner) - 1) : 0.0;
  }

  // scan that chunk in index order: lane l owns GPL contiguous groups of 4 elements,
  // whose weights stay in registers
  const bool no_q = use_p || qrow == nullptr;
  const float iz = use_p ? invZp : invZ;
  const int k0 = cstar * kDrawChunk;
  const int ng = min(kDrawChunk, P.V - k0) / 4;
  float w[GPL][4];
  float gsum[GPL];
  double lane_tot = 0.0;
#pragma unroll
  for (int j = 0; j < GPL; ++j) {
    const int g = lane * GPL + j;
    gsum[j] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) w[j][e] = 0.f;
    if (g < ng) {
      const GL lw = __ldg(reinterpret_cast<const GL*>(lrow + k0) + g);
      const float4 q4 = no_q ? make_float4(0.f, 0.f, 0.f, 0.f) : __ldg(reinterpret_cast<const float4*>(qrow + k0) + g);
      gsum[j] = group_weights<T>(lw, q4, mJ, c, iz, no_q, w[j]);
      lane_tot += static_cast<double>(gsum[j]);
    }
  }
  int last_pos = -1;
#pragma unroll
  for (int j = 0; j < GPL; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (w[j][e] > 0.f) last_pos = k0 + 4 * (lane * GPL + j) + e;
  const double gincl = warp_incl_scan(lane_tot, lane);
  const unsigned ghit = __ballot_sync(0xffffffffu, base + gincl > target);
  int y = -1;
  if (ghit) {
    const int fl = __ffs(ghit) - 1;
    if (lane == fl) {
      double pre = base + (gincl - lane_tot);
#pragma unroll
      for (int j = 0; j < GPL; ++j) {
        if (y < 0 && pre + static_cast<double>(gsum[j]) > target) {
          float run = 0.f;
          int lastp = -1;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            run += w[j][e];
            if (w[j][e] > 0.f) lastp = k0 + 4 * (lane * GPL + j) + e;
            if (y < 0 && pre + static_cast<double>(run) > target) y = k0 + 4 * (lane * GPL + j) + e;
          }
          if (y < 0) y = lastp;
        }
        pre += static_cast<double>(gsum[j]);
      }
    }
    y = __shfl_sync(0xffffffffu, y, fl);
  }
  if (y < 0) y = warp_max_int(last_pos);  // rounding put u * S at or past the chunk's end
  return y;
}

template <typename T>
__global__ void __launch_bounds__(32) chain_finish_kernel(const ChainParams P) {
  grid_launch_dependents();
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x;
  SeqState st;
  st.meta = __ldcg(&P.ws.seq[b].meta);
  st.row = __ldcg(&P.ws.seq[b].row);
  if (st.meta.y != 1) return;
  const int R = P.gamma + 1;
  const int J = st.meta.x;
  const float* dm = P.ws.draw_mass + static_cast<int64_t>(b) * P.nchd;
  int32_t* tok_out = P.out_tokens + static_cast<int64_t>(b) * R;
  const T* lrow = static_cast<const T*>(P.logits) + (static_cast<int64_t>(b) * R + J) * P.V;
  const float* qrow = (J < P.gamma) ? P.q + (static_cast<int64_t>(b) * P.gamma + J) * P.V : nullptr;
  const float invZ = 1.f / st.row.y;
  bool zr = false;
  const int y = draw_from_masses<T>(P, dm, lrow, qrow, st.row.x, st.row.z, invZ, invZ, st.row.w, lane, zr);
  if (y < 0) {  // a bad draft probability in the drawn row
    if (lane < R) tok_out[lane] = -1;
    if (lane < P.gamma && P.out_p_draft) P.out_p_draft[static_cast<int64_t>(b) * P.gamma + lane] = kNaN;
    if (lane == 0) {
      P.out_J[b] = -1;
      if (P.out_status) P.out_status[b] = st.meta.z | SPECDEC_STATUS_BAD_PROB;
    }
    return;
  }
  if (lane == 0) {
    tok_out[J] = y;
    if (zr && P.out_status) P.out_status[b] = st.meta.z | SPECDEC_STATUS_ZERO_RESIDUAL;
  }
}

// ---------------------------------------------------------------------------------
// Block verification (Art of Guessing, "Block verification", Sun et al.): the same
// statistics pass, then
//   block decide  one CTA per sequence: every row's (m, Z) and argmax, p_k(x_k), the
//                 running weights w_{k+1} = min(1, w_k p_k(x_k) / q_k(x_k)) (w_0 = 1),
//                 every input checked; lists all gamma + 1 rows for the mass pass with
//                 their weights folded into the scale: (w_k p_k - q_k)+ (q_gamma = 0).
//   mass pass     the draw kernel above, over every listed row.
//   block finish  one CTA per sequence: mass_k per row (fp64), survival_k =
//                 mass_k / (mass_k + 1 - w_k) (1 if w_k = 1), n = the longest prefix k
//                 with u[k-1] <= survival_k, and the inverse-CDF draw from row n.
// ---------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kDecideThreads) block_decide_kernel(const ChainParams P) {
  __shared__ float s_m[kStreamMaxRows], s_Z[kStreamMaxRows];
  __shared__ int s_z[kStreamMaxRows];
  grid_launch_dependents();
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = P.gamma + 1;
  const int nch = P.nch;
  const float Tb = P.greedy_only ? 0.f : __ldg(P.temps + b);
  const bool greedy = P.greedy_only || is_greedy(Tb);
  const float c = greedy ? 0.f : kLog2e / Tb;

  // inputs (lane i: position i; lane gamma: the draw's uniform), before the wait
  int x = -1, tok_err = 0, u_err = 0;
  float lx = 0.f, qx = 0.f, ux = 0.f;
  if (warp == 0) {
    if (lane < P.gamma) {
      x = __ldg(P.drafts + static_cast<int64_t>(b) * P.gamma + lane);
      if (x < 0 || x >= P.V) {
        tok_err = SPECDEC_STATUS_BAD_TOKEN;
      } else if (!greedy) {
        lx = Elem<T>::load(static_cast<const T*>(P.logits) + (static_cast<int64_t>(b) * R + lane) * P.V, x);
        qx = __ldg(P.q + (static_cast<int64_t>(b) * P.gamma + lane) * P.V + x);
      }
    }
    if (!greedy && lane < R) {
      ux = __ldg(P.u + static_cast<int64_t>(b) * R + lane);
      if (!(ux >= 0.f && ux < 1.f)) u_err = SPECDEC_STATUS_BAD_UNIFORM;
    }
  }
  grid_dependency_wait();

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

  float m = -kInf, Z = 0.f;
  int z = INT_MAX, row_err = 0;
  if (lane < R) {
    m = s_m[lane];
    Z = s_Z[lane];
    z = s_z[lane];
    if (!(m == m) || m == kInf) row_err = SPECDEC_STATUS_BAD_LOGIT;
    else if (m == -kInf) row_err = SPECDEC_STATUS_EMPTY_ROW;
  }
  // every row, draft and uniform is read by the rule: every error is reported
  int err = __reduce_or_sync(0xffffffffu, row_err | tok_err | u_err);
  const bool bad_T = !P.greedy_only && !(Tb - Tb == 0.f);
  if (bad_T) err = SPECDEC_STATUS_BAD_TEMPERATURE;
  int32_t* tok_out = P.out_tokens + static_cast<int64_t>(b) * R;
  float* pd_out = P.out_p_draft ? P.out_p_draft + static_cast<int64_t>(b) * P.gamma : nullptr;

  if (greedy || bad_T) {
    // greedy matching (a one-hot target reduces the block rule to it)
    const bool miss = lane < P.gamma && x != z;
    const unsigned mm = __ballot_sync(0xffffffffu, miss);
    const int J = err ? -1 : (mm ? __ffs(mm) - 1 : P.gamma);
    const int zJ = __shfl_sync(0xffffffffu, z, J < 0 ? 0 : J);
    if (lane < R) tok_out[lane] = (J < 0) ? -1 : (lane < J ? x : (lane == J ? zJ : -1));
    if (lane < P.gamma && pd_out) pd_out[lane] = kNaN;
    if (lane == 0) {
      P.out_J[b] = J;
      if (P.out_status) P.out_status[b] = err;
      SeqState sq;
      sq.meta = make_int4(J, 0, err, 0);
      sq.row = make_float4(0.f, 0.f, 0.f, 0.f);
      P.ws.seq[b] = sq;
    }
    return;
  }

  // p_k(x_k), the ratios and the running weights (one serial pass over the positions)
  float px = kNaN;
  int warn = 0;
  float ratio = 0.f;
  if (lane < P.gamma && !tok_err) {
    px = ex2((lx - m) * c) / Z;
    if (qx == 0.f) {
      warn = SPECDEC_STATUS_ZERO_Q;
      ratio = px > 0.f ? kInf : 0.f;
    } else {
      ratio = px / qx;
    }
  }
  warn = __reduce_or_sync(0xffffffffu, warn);
  float w = 1.f, wk = 1.f;  // wk: this lane's w_lane
  for (int k = 0; k < P.gamma; ++k) {
    const float rk = __shfl_sync(0xffffffffu, ratio, k);
    w = (w == 0.f) ? 0.f : fminf(1.f, w * rk);
    if (lane == k + 1) wk = w;
  }
  if (lane < P.gamma && pd_out) pd_out[lane] = err ? kNaN : px;
  if (lane < R) P.ws.block_rows[static_cast<int64_t>(b) * R + lane] = make_float4(m, Z, wk, 0.f);
  // Rows for the mass pass: the gamma rows with q always (their q rows are checked even
  // when the sequence already failed), the bonus row only for a clean sequence.
  const int nent = err ? P.gamma : R;
  unsigned base = 0;
  if (lane == 0) base = atomicAdd(P.ws.draw_count, static_cast<unsigned>(nent));
  base = __shfl_sync(0xffffffffu, base, 0);
  if (lane < nent) {
    DrawEntry d;
    d.loc = make_int4(b, lane, b * R + lane, 0);
    d.row = make_float4(m, c, wk / Z, 0.f);
    P.ws.draw_list[base + lane] = d;
  }
  if (lane == 0) {
    SeqState sq;
    sq.meta = make_int4(-1, 2, err | warn, 0);
    sq.row = make_float4(0.f, 0.f, c, 0.f);
    P.ws.seq[b] = sq;
  }
}

template <typename T>
__global__ void __launch_bounds__(kDecideThreads) block_finish_kernel(const ChainParams P) {
  __shared__ double s_mass[kStreamMaxRows];
  grid_launch_dependents();
  grid_dependency_wait();
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  SeqState st;
  st.meta = __ldcg(&P.ws.seq[b].meta);
  st.row = __ldcg(&P.ws.seq[b].row);
  if (st.meta.y != 2) return;
  const int R = P.gamma + 1;
  const int nchd = P.nchd;
  int status = st.meta.z;
  if (__ldcg(P.ws.qbad + b)) status |= SPECDEC_STATUS_BAD_PROB;
  int32_t* tok_out = P.out_tokens + static_cast<int64_t>(b) * R;
  if (status & SPECDEC_STATUS_ERROR_MASK) {  // errors only: warnings describe a clean round
    status &= SPECDEC_STATUS_ERROR_MASK;
    if (warp == 0) {
      if (lane < R) tok_out[lane] = -1;
      if (lane < P.gamma && P.out_p_draft) P.out_p_draft[static_cast<int64_t>(b) * P.gamma + lane] = kNaN;
      if (lane == 0) {
        P.out_J[b] = -1;
        if (P.out_status) P.out_status[b] = status;
      }
    }
    return;
  }
  // mass_k of every row (fp64, fixed order: lane-contiguous runs, then the warp)
  for (int k = warp; k < R; k += kDecideThreads / 32) {
    const float* dm = P.ws.draw_mass + (static_cast<int64_t>(b) * R + k) * nchd;
    const int cpl = (nchd + 31) / 32;
    const int q0 = min(lane * cpl, nchd), q1 = min(q0 + cpl, nchd);
    double mine = 0.0;
    for (int q = q0; q < q1; ++q) mine += static_cast<double>(__ldcg(dm + q));
    const double tot = warp_incl_scan(mine, lane);
    if (lane == 31) s_mass[k] = tot;
  }
  __syncthreads();
  if (warp != 0) return;
  // survival of every prefix and the longest surviving one
  float4 br = make_float4(0.f, 1.f, 1.f, 0.f);
  if (lane < R) br = __ldcg(P.ws.block_rows + static_cast<int64_t>(b) * R + lane);
  const double wk = static_cast<double>(br.z);
  bool survived = false;
  if (lane >= 1 && lane < R) {
    const double mass = s_mass[lane];
    const double surv = (wk < 1.0) ? mass / (mass + 1.0 - wk) : 1.0;
    const float uk = __ldg(P.u + static_cast<int64_t>(b) * R + lane - 1);
    survived = static_cast<double>(uk) <= surv;
  }
  const unsigned sv = __ballot_sync(0xffffffffu, survived);
  const int n = sv ? 31 - __clz(sv) : 0;
  const float mN = __shfl_sync(0xffffffffu, br.x, n), zN = __shfl_sync(0xffffffffu, br.y, n);
  const float wN = __shfl_sync(0xffffffffu, br.z, n);
  const float c = st.row.z;
  const T* lrow = static_cast<const T*>(P.logits) + (static_cast<int64_t>(b) * R + n) * P.V;
  const float* qrow = (n < P.gamma) ? P.q + (static_cast<int64_t>(b) * P.gamma + n) * P.V : nullptr;
  const float uG = __ldg(P.u + static_cast<int64_t>(b) * R + P.gamma);
  bool zr = false;
  const int y = draw_from_masses<T>(P, P.ws.draw_mass + (static_cast<int64_t>(b) * R + n) * nchd, lrow, qrow, mN,
                                    c, wN / zN, 1.f / zN, uG, lane, zr);
  const int x = (lane < P.gamma) ? __ldg(P.drafts + static_cast<int64_t>(b) * P.gamma + lane) : -1;
  if (lane < R) tok_out[lane] = lane < n ? x : (lane == n ? y : -1);
  if (lane == 0) {
    P.out_J[b] = n;
    if (P.out_status) P.out_status[b] = status | (zr ? SPECDEC_STATUS_ZERO_RESIDUAL : 0);
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
  constexpr int smem = draw_smem_bytes<T>();
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

cudaError_t launch_block_decide(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream) {
  if (ldt == SPECDEC_BF16)
    return launch_kernel(block_decide_kernel<uint16_t>, dim3(P.B), dim3(kDecideThreads), 0, stream, 1, P);
  return launch_kernel(block_decide_kernel<float>, dim3(P.B), dim3(kDecideThreads), 0, stream, 1, P);
}

cudaError_t launch_block_finish(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream) {
  if (ldt == SPECDEC_BF16)
    return launch_kernel(block_finish_kernel<uint16_t>, dim3(P.B), dim3(kDecideThreads), 0, stream, 1, P);
  return launch_kernel(block_finish_kernel<float>, dim3(P.B), dim3(kDecideThreads), 0, stream, 1, P);
}

cudaError_t launch_chain_stream_finish(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream) {
  if (ldt == SPECDEC_BF16)
    return launch_kernel(chain_finish_kernel<uint16_t>, dim3(P.B), dim3(32), 0, stream, 1, P);
  return launch_kernel(chain_finish_kernel<float>, dim3(P.B), dim3(32), 0, stream, 1, P);
}

}  // namespace specdec
