// Device pieces shared by the streaming verification kernels (chain_stream.cu) and the
// single-read block-verification kernel (block_fused.cu): warp reductions, the merge of
// (max, normaliser, argmax) row summaries, the residual weights of 4-element groups, the
// draft-probability check, and the inverse-CDF draw from a row's chunk masses.
#pragma once

#include <climits>

#include "specdec_device.cuh"
#include "specdec_internal.h"

namespace specdec {
namespace {

constexpr uint32_t kNegInfBf16x2 = 0xFF80FF80u;
constexpr float kNaN = __builtin_nanf("");

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


// The summary of one 4 KB chunk of logits held as 16-byte vectors, VPL per lane (lane
// l holds vectors l, l + 32, ...; nv vectors are valid, the rest read as -inf): its maximum
// m, then for a sampled row the sum of 2^((l - m) c) (packed f32x2 arithmetic, one ex2 per
// element), or for a greedy row the lowest index of the maximum (ch = the chunk's index in
// its row).  Returns (m, Z, argmax bits, 0), the same in every lane.
template <typename T>
__device__ __forceinline__ float4 chunk_summary(const uint4 (&w)[kStatsChunkBytes / 16 / 32], int nv, uint32_t ch,
                                                bool greedy, float c) {
  constexpr int VEC = Vec<T>::n;
  constexpr int VPL = kStatsChunkBytes / 16 / 32;
  constexpr int EPC = kStatsChunkBytes / static_cast<int>(sizeof(T));  // elements per chunk
  const int lane = threadIdx.x & 31;
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
  return make_float4(m, Z, __int_as_float(z), 0.f);
}

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


// Mass of chunk q of the drawn row: the draw kernel's residual mass, or (zero-residual
// fallback) the mass of p itself, recomputed here.
template <typename T, int CH>
__device__ __forceinline__ float chunk_mass(int V, const float* dm, bool use_p, const T* lrow, int q, float mJ,
                                            float c, float invZ) {
  if (!use_p) return __ldcg(dm + q);
  using GL = typename Group<T>::L;
  const int k0 = q * CH;
  const int ng = min(CH, V - k0) / 4;
  float acc = 0.f;
  for (int g = 0; g < ng; ++g) {
    float w[4];
    acc += group_weights<T>(__ldg(reinterpret_cast<const GL*>(lrow + k0) + g), make_float4(0.f, 0.f, 0.f, 0.f),
                            mJ, c, invZ, true, w);
  }
  return acc;
}

// Index-order scan of chunk cstar (CH elements) of one row for the smallest k with
// C_k > target, where C is the running weight (residual (p - q)+ with p = 2^((l - m)c) * iz,
// or p alone when no_q) and `base` is the mass before the chunk.  Lane l owns GPL
// contiguous groups of 4 elements, whose weights stay in registers.  Rounding that puts the
// target at or past the chunk's end gives the chunk's last positive-weight element.
template <typename T, int CH>
__device__ int scan_chunk(int V, const T* lrow, const float* qrow, float mJ, float c, float iz, bool no_q, int cstar,
                          double base, double target, int lane) {
  using GL = typename Group<T>::L;
  constexpr int GPL = CH / 4 / 32;
  const int k0 = cstar * CH;
  const int ng = min(CH, V - k0) / 4;
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

// The inverse-CDF draw from one row's masses of CH-element chunks (one warp): the chunk whose fp64
// running mass first exceeds u * S, then an index-order scan of that chunk for the
// smallest k with C_k > u * S.  invZ scales the weights the masses were made with
// ((p - q)+ with p = 2^((l - m)c) * invZ, q == nullptr for none); a total of zero (possible
// only through rounding) draws from p itself, whose chunk masses are recomputed with
// invZp (dm == nullptr: no masses, draw from p).  Returns the token, or -1 when a mass is
// NaN (a bad draft probability).
template <typename T, int CH>
__device__ int draw_from_masses(int V, int nchd, const float* dm, const T* lrow, const float* qrow, float mJ,
                                float c, float invZ, float invZp, float u, int lane, bool& zero_residual) {
  static_assert(CH % 128 == 0, "a chunk is whole 4-element groups of every lane");
  constexpr int CPL = 16;                   // chunk masses per lane kept in registers
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
    for (int j = 0; j < CPL; ++j) wq[j] = (dm != nullptr && c0 + j < c1) ? __ldcg(dm + c0 + j) : 0.f;
#pragma unroll
    for (int j = 0; j < CPL; ++j)
      if (j < c1 - c0) mine += static_cast<double>(wq[j]);
  } else {
    for (int q = c0; q < c1 && dm != nullptr; ++q) mine += static_cast<double>(__ldcg(dm + q));
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
        wq[j] = (j < c1 - c0) ? chunk_mass<T, CH>(V, dm, true, lrow, c0 + j, mJ, c, invZp) : 0.f;
        mine += static_cast<double>(wq[j]);
      }
    } else {
      for (int q = c0; q < c1; ++q) mine += static_cast<double>(chunk_mass<T, CH>(V, dm, true, lrow, q, mJ, c, invZp));
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
        const double w = static_cast<double>(chunk_mass<T, CH>(V, dm, use_p, lrow, q, mJ, c, invZp));
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

  const bool no_q = use_p || qrow == nullptr;
  return scan_chunk<T, CH>(V, lrow, qrow, mJ, c, use_p ? invZp : invZ, no_q, cstar, base, target, lane);
}

}  // namespace
}  // namespace specdec
