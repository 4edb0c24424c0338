// Chain verification that reads only the rows a round needs.
//
// SD 20.5, "A whole round of speculative sampling": the one-token rule is applied to the
// drafts left to right and the round stops at the first rejection; the drafts after it
// are discarded, so their target rows are never needed.  This kernel follows that order
// literally.  Each CTA (one per SM, persistent) holds kSeqGroups groups of warps; a group
// takes whole sequences from a shared counter and, for each:
//
//   row i = 0, 1, ...  stream the row through the group's bulk-copy pipelines (every warp
//                      keeps three cp.async.bulk copies in flight on mbarriers); each lane
//                      keeps a running maximum and sum of 2^((l - m) * log2(e) / T) (or the
//                      lowest index of the maximum for a greedy sequence); the group merges
//                      them and tests draft i: accept iff u_i * q_i(x_i) < p_i(x_i)
//                      (greedy: x_i == argmax).  A rejection, or row gamma, ends the loop.
//   draw               for a sampled sequence, one more pass over the last row read (J)
//                      and q row J: residual weights (p_J - q_J)+ (q == 0 for the bonus
//                      row; SD 20.5, "The speculative sampling rule") summed per 512-element
//                      chunk in shared memory, then an fp64 prefix over the chunks and an
//                      index-order scan of the chosen chunk for the smallest k with
//                      C_k > u * S.
//
// Everything a sequence needs stays inside its group: no grid-wide synchronisation, no
// fences.  The only shared datum is the sequence counter (cleared by the host per call).

#include <climits>

#include "specdec_device.cuh"
#include "specdec_internal.h"

namespace specdec {

namespace {

constexpr uint32_t kNegInfBf16x2 = 0xFF80FF80u;
constexpr float kNaN = __builtin_nanf("");
constexpr int kWarpsPerGroup = kSeqWarps / kSeqGroups;
constexpr int kGroupThreads = kWarpsPerGroup * 32;

__device__ __forceinline__ bool is_greedy(float T) { return !(T >= SPECDEC_GREEDY_TEMPERATURE); }

// Barrier over the threads of one group (named barriers 1.., 0 stays __syncthreads).
__device__ __forceinline__ void group_sync(int group) {
  asm volatile("bar.sync %0, %1;" ::"r"(group + 1), "r"(kGroupThreads) : "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
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

// (max, normaliser, lowest argmax) of a part of a row, and the merge of two parts.
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

template <typename T> struct Vec;
template <> struct Vec<uint16_t> { static constexpr int n = 8; };
template <> struct Vec<float> { static constexpr int n = 4; };

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

// Residual (or target) weights of 4 consecutive elements and their fp32 running sum in
// index order; the chunk masses and the final scan both use it.
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

// Shared state of one group.
struct GroupShared {
  RowSum wsum[kWarpsPerGroup];  // per-warp row summaries
  float mass[kSeqMaxDrawChunks];  // draw: residual mass per chunk
  float4 row;                   // merged row (m, Z, argmax bits, 0)
  int b;                        // current sequence (or >= B: done)
  int stop;                     // decision broadcast
  int qbad;                     // a bad draft probability in the drawn row
  int y;                        // drawn token
};

// One warp's bulk-copy pipeline: kSeqStages stages of kSeqChunkBytes in shared memory.
// `k` counts completed stages and `issued` issued ones, over the kernel's lifetime.
struct Pipe {
  unsigned char* buf;
  uint64_t* bar;
  uint32_t k = 0, issued = 0;
  bool ok = true;  // false once a bounded wait gave up

  __device__ __forceinline__ unsigned char* stage(uint32_t i) { return buf + (i % kSeqStages) * kSeqChunkBytes; }
  __device__ __forceinline__ uint64_t* sbar(uint32_t i) { return bar + (i % kSeqStages); }
  // Issue one copy group (one or two copies totalling `bytes`) into the next stage.
  __device__ __forceinline__ void issue(const void* a, uint32_t na, const void* b, uint32_t nb, int off_b) {
    uint64_t* br = sbar(issued);
    unsigned char* dst = stage(issued);
    mbar_expect_tx(br, na + nb);
    bulk_copy_g2s(dst, a, na, br);
    if (nb) bulk_copy_g2s(dst + off_b, b, nb, br);
  }
  __device__ __forceinline__ bool wait() { return mbar_wait(sbar(k), (k / kSeqStages) & 1u); }
};

// ---------------------------------------------------------------------------------
// One logits row: per-lane running summary across the warp's chunks, group merge.
// ---------------------------------------------------------------------------------
template <typename T>
__device__ RowSum row_pass(const T* lrow, int V, bool greedy, float c, Pipe& pp, GroupShared& gs,
                           int group, int gwarp, int lane, unsigned* error) {
  constexpr int VEC = Vec<T>::n;
  constexpr int VPL = kSeqChunkBytes / 16 / 32;
  constexpr int EPC = kSeqChunkBytes / static_cast<int>(sizeof(T));
  const int64_t row_bytes = static_cast<int64_t>(V) * sizeof(T);
  const int nch = static_cast<int>((row_bytes + kSeqChunkBytes - 1) / kSeqChunkBytes);
  const char* base = reinterpret_cast<const char*>(lrow);
  auto chunk_bytes = [&](int ch) -> uint32_t {
    return static_cast<uint32_t>(min(static_cast<int64_t>(kSeqChunkBytes), row_bytes - static_cast<int64_t>(ch) * kSeqChunkBytes));
  };
  // this warp's chunks: gwarp, gwarp + W, ...
  int next = gwarp;
  if (pp.ok) {
    for (int s = 0; s < kSeqStages && next < nch; ++s, next += kWarpsPerGroup) {
      if (lane == 0) pp.issue(base + static_cast<int64_t>(next) * kSeqChunkBytes, chunk_bytes(next), nullptr, 0, 0);
      ++pp.issued;
    }
  }
  float ml = -kInf, Zl = 0.f;
  int zl = INT_MAX;
  // After a bounded wait gives up (never expected) this warp stops copying but keeps
  // taking part in its group's barriers; the kernel records the failure.
  for (int ch = gwarp; ch < nch && pp.ok; ch += kWarpsPerGroup) {
    if (!pp.wait()) {
      if (lane == 0) atomicOr(error, 1u);
      pp.ok = false;
      break;
    }
    const int nv = static_cast<int>(chunk_bytes(ch) / 16);
    const uint4* vb = reinterpret_cast<const uint4*>(pp.stage(pp.k));
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
    ++pp.k;
    if (next < nch) {  // refill the stage just read with this warp's next chunk
      if (lane == 0) {
        fence_proxy_async_smem();
        pp.issue(base + static_cast<int64_t>(next) * kSeqChunkBytes, chunk_bytes(next), nullptr, 0, 0);
      }
      ++pp.issued;
      next += kWarpsPerGroup;
    }
    // chunk maximum of this lane
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
    if (greedy) {
      // strictly larger maximum: locate its first index in this chunk (earlier chunks keep ties)
      if (mt > ml || (mt != mt && ml == ml)) {
        int idx = INT_MAX;
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
          const uint32_t ww[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            float v;
            if constexpr (sizeof(T) == 2) v = (e & 1) ? bf16_hi(ww[e >> 1]) : bf16_lo(ww[e >> 1]);
            else v = __uint_as_float(ww[e]);
            if (idx == INT_MAX && v == mt && lane + 32 * j < nv) idx = ch * EPC + (lane + 32 * j) * VEC + e;
          }
        }
        ml = mt;
        zl = idx;
      }
    } else {
      // online softmax: rescale the running sum when the maximum grows
      const float mn = max_nan(ml, mt);
      if (mn > -kInf) {
        if (mn != ml) Zl = (ml > -kInf) ? Zl * ex2((ml - mn) * c) : 0.f;
        ml = mn;
        const unsigned long long m2 = f2pack(ml, ml), c2 = f2pack(c, c);
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
        Zl += a0 + a1;
      } else {
        ml = mn;  // NaN propagates; -inf stays
      }
    }
  }
  RowSum r;
  r.m = ml;
  r.Z = Zl;
  r.z = zl;
  r = warp_merge(r, c);
  if (lane == 0) gs.wsum[gwarp] = r;
  group_sync(group);
  if (gwarp == 0) {
    RowSum t;
    t.m = -kInf;
    t.Z = 0.f;
    t.z = INT_MAX;
    if (lane < kWarpsPerGroup) t = gs.wsum[lane];
    t = warp_merge(t, c);
    if (lane == 0) gs.row = make_float4(t.m, t.Z, __int_as_float(t.z), 0.f);
  }
  group_sync(group);
  const float4 f = gs.row;
  RowSum out;
  out.m = f.x;
  out.Z = f.y;
  out.z = __float_as_int(f.z);
  return out;
}

// ---------------------------------------------------------------------------------
// The draw over row J: chunk masses (group), then the inverse-CDF search (first warp).
// ---------------------------------------------------------------------------------
template <typename T>
__device__ int draw_pass(const ChainParams& P, const T* lrow, const float* qrow, float mJ, float c,
                         float invZ, float u, Pipe& pp, GroupShared& gs, int group, int gwarp, int lane,
                         bool& zero_residual, bool& bad_q) {
  using GL = typename Group<T>::L;
  constexpr int LB = kSeqDrawChunk * static_cast<int>(sizeof(T));
  constexpr int GPL = kSeqDrawChunk / 4 / 32;
  const int V = P.V;
  const int nchd = (V + kSeqDrawChunk - 1) / kSeqDrawChunk;
  int next = gwarp;
  auto issue = [&](int cd) {
    const int n = min(kSeqDrawChunk, V - cd * kSeqDrawChunk);
    const int64_t off = static_cast<int64_t>(cd) * kSeqDrawChunk;
    if (lane == 0)
      pp.issue(lrow + off, static_cast<uint32_t>(n) * sizeof(T), qrow ? qrow + off : nullptr,
               qrow ? static_cast<uint32_t>(n) * 4u : 0u, LB);
    ++pp.issued;
  };
  if (pp.ok)
    for (int s = 0; s < kSeqStages && next < nchd; ++s, next += kWarpsPerGroup) issue(next);
  float qmx = 0.f, qmn = 0.f;
  for (int cd = gwarp; cd < nchd && pp.ok; cd += kWarpsPerGroup) {
    if (!pp.wait()) {
      if (lane == 0) atomicOr(P.ws.error, 1u);
      pp.ok = false;
      break;
    }
    const int ng = min(kSeqDrawChunk, V - cd * kSeqDrawChunk) / 4;
    const unsigned char* sb = pp.stage(pp.k);
    GL lw[GPL];
    float4 qv[GPL];
#pragma unroll
    for (int j = 0; j < GPL; ++j) {
      const int g = lane + 32 * j;
      if (g < ng) {
        lw[j] = reinterpret_cast<const GL*>(sb)[g];
        qv[j] = qrow ? reinterpret_cast<const float4*>(sb + LB)[g] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    __syncwarp();
    ++pp.k;
    if (next < nchd) {
      if (lane == 0) fence_proxy_async_smem();
      issue(next);
      next += kWarpsPerGroup;
    }
    float sr = 0.f;
#pragma unroll
    for (int j = 0; j < GPL; ++j) {
      if (lane + 32 * j < ng) {
        float w[4];
        sr += group_weights<T>(lw[j], qv[j], mJ, c, invZ, qrow == nullptr, w);
        qmx = max_nan(qmx, max_nan(max_nan(qv[j].x, qv[j].y), max_nan(qv[j].z, qv[j].w)));
        qmn = fminf(qmn, fminf(fminf(qv[j].x, qv[j].y), fminf(qv[j].z, qv[j].w)));
      }
    }
    sr = warp_sum(sr);
    if (lane == 0) gs.mass[cd] = sr;
  }
  const bool mybad = !(qmx < kInf) || qmn < 0.f;
  if (lane == 0 && gwarp == 0) gs.qbad = 0;
  group_sync(group);
  if (__any_sync(0xffffffffu, mybad) && lane == 0) atomicOr(&gs.qbad, 1);
  group_sync(group);
  bad_q = gs.qbad != 0;
  zero_residual = false;
  if (bad_q) return -1;

  // total residual mass; zero (possible only through rounding) falls back to p itself
  if (gwarp == 0) {
    double tot = 0.0;
    for (int q = lane; q < nchd; q += 32) tot += static_cast<double>(gs.mass[q]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    if (lane == 0) gs.stop = !(tot > 0.0);
  }
  group_sync(group);
  zero_residual = gs.stop != 0;
  if (zero_residual) {
    for (int cd = gwarp; cd < nchd; cd += kWarpsPerGroup) {  // rare: masses of p itself
      const int ng = min(kSeqDrawChunk, V - cd * kSeqDrawChunk) / 4;
      float sr = 0.f;
      for (int g = lane; g < ng; g += 32) {
        float w[4];
        sr += group_weights<T>(__ldg(reinterpret_cast<const GL*>(lrow + static_cast<int64_t>(cd) * kSeqDrawChunk) + g),
                               make_float4(0.f, 0.f, 0.f, 0.f), mJ, c, invZ, true, w);
      }
      sr = warp_sum(sr);
      if (lane == 0) gs.mass[cd] = sr;
    }
    group_sync(group);
  }
  const bool no_q = zero_residual || qrow == nullptr;

  // inverse CDF: chunk by fp64 prefix, then an index-order scan inside the chunk
  if (gwarp == 0) {
    const int cpl = (nchd + 31) / 32;
    const int c0 = min(lane * cpl, nchd), c1 = min(c0 + cpl, nchd);
    double mine = 0.0;
    for (int q = c0; q < c1; ++q) mine += static_cast<double>(gs.mass[q]);
    const double incl = warp_incl_scan(mine, lane);
    const double S = __shfl_sync(0xffffffffu, incl, 31);
    const double target = static_cast<double>(u) * S;
    int cstar = -1, lastpos = -1;
    double base = 0.0, prelast = 0.0, pre = incl - mine;
    for (int q = c0; q < c1; ++q) {
      const double w = static_cast<double>(gs.mass[q]);
      if (w > 0.0) { lastpos = q; prelast = pre; }
      if (cstar < 0 && pre + w > target) { cstar = q; base = pre; }
      pre += w;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, cstar >= 0);
    if (hit) {
      const int fl = __ffs(hit) - 1;
      cstar = __shfl_sync(0xffffffffu, cstar, fl);
      base = __shfl_sync(0xffffffffu, base, fl);
    } else {  // rounding put u * S at or past the end: last chunk with mass
      const int best = warp_max_int(lastpos);
      const unsigned owner = __ballot_sync(0xffffffffu, lastpos == best && best >= 0);
      cstar = best < 0 ? 0 : best;
      base = owner ? __shfl_sync(0xffffffffu, prelast, __ffs(owner) - 1) : 0.0;
    }
    const int k0 = cstar * kSeqDrawChunk;
    const int ng = min(kSeqDrawChunk, V - k0) / 4;
    float w[GPL][4], gsum[GPL];
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
        gsum[j] = group_weights<T>(lw, q4, mJ, c, invZ, no_q, w[j]);
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
        double p2 = base + (gincl - lane_tot);
#pragma unroll
        for (int j = 0; j < GPL; ++j) {
          if (y < 0 && p2 + static_cast<double>(gsum[j]) > target) {
            float run = 0.f;
            int lastp = -1;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              run += w[j][e];
              if (w[j][e] > 0.f) lastp = k0 + 4 * (lane * GPL + j) + e;
              if (y < 0 && p2 + static_cast<double>(run) > target) y = k0 + 4 * (lane * GPL + j) + e;
            }
            if (y < 0) y = lastp;
          }
          p2 += static_cast<double>(gsum[j]);
        }
      }
      y = __shfl_sync(0xffffffffu, y, fl);
    }
    if (y < 0) y = warp_max_int(last_pos);
    if (lane == 0) gs.y = y;
  }
  group_sync(group);
  return gs.y;
}

// ---------------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kSeqWarps * 32, 1) chain_seq_kernel(const ChainParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t bars[kSeqWarps][kSeqStages];
  __shared__ GroupShared gshared[kSeqGroups];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int group = warp / kWarpsPerGroup, gwarp = warp % kWarpsPerGroup;
  GroupShared& gs = gshared[group];
  Pipe pp;
  pp.buf = smem + static_cast<size_t>(warp) * kSeqStages * kSeqChunkBytes;
  pp.bar = bars[warp];
  if (lane == 0) {
    for (int s = 0; s < kSeqStages; ++s) mbar_init(&pp.bar[s], 1);
    mbar_fence_init();
  }
  __syncwarp();
  const int R = P.gamma + 1;

  for (;;) {
    if (threadIdx.x % kGroupThreads == 0) gs.b = static_cast<int>(atomicAdd(P.ws.draw_count, 1u));
    group_sync(group);
    const int b = gs.b;
    if (b >= P.B) break;
    const float Tb = P.greedy_only ? 0.f : __ldg(P.temps + b);
    const bool greedy = P.greedy_only || is_greedy(Tb);
    const float c = greedy ? 0.f : kLog2e / Tb;
    const bool bad_T = !P.greedy_only && !(Tb - Tb == 0.f);

    // The group's first warp holds position i in lane i: its draft, the logit and q at
    // the draft, and its uniform (lane gamma: the draw's uniform), fetched up front.
    int x = -1, tok_err = 0, qu_err = 0;
    float lx = 0.f, qx = 0.f, ux = 0.f, px = kNaN;
    if (gwarp == 0) {
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

    // rows in order until the first error or rejection
    int J = -1, st = bad_T ? SPECDEC_STATUS_BAD_TEMPERATURE : 0, warn = 0;
    RowSum rs;
    rs.m = 0.f;
    rs.Z = 1.f;
    rs.z = 0;
    if (!bad_T) {
      for (int i = 0; i < R; ++i) {
        rs = row_pass<T>(static_cast<const T*>(P.logits) + (static_cast<int64_t>(b) * R + i) * P.V, P.V, greedy, c,
                         pp, gs, group, gwarp, lane, P.ws.error);
        if (gwarp == 0) {
          int err = 0;
          if (!(rs.m == rs.m) || rs.m == kInf) err = SPECDEC_STATUS_BAD_LOGIT;
          else if (rs.m == -kInf) err = SPECDEC_STATUS_EMPTY_ROW;
          else if (i < P.gamma) err = __shfl_sync(0xffffffffu, tok_err ? tok_err : qu_err, i);
          int stop = 0;
          if (err) {
            st |= err;
            stop = 2;
          } else if (i == P.gamma) {
            stop = 1;
          } else {
            bool acc = false;
            float pxi = kNaN;
            if (lane == i) {
              if (greedy) {
                acc = (x == rs.z);
              } else {
                pxi = ex2((lx - rs.m) * c) / rs.Z;
                if (qx == 0.f) {
                  warn |= SPECDEC_STATUS_ZERO_Q;
                  acc = pxi > 0.f;
                } else {
                  acc = ux * qx < pxi;
                }
                px = pxi;
              }
            }
            stop = __shfl_sync(0xffffffffu, acc ? 0 : 1, i);
          }
          if (lane == 0) gs.stop = stop;
        }
        group_sync(group);
        const int stop = gs.stop;
        if (stop) {
          J = (stop == 2) ? -1 : i;  // -1: an error ended the round
          break;
        }
        group_sync(group);  // gs.stop is rewritten by the next row's decision
      }
    }
    if (gwarp == 0) {
      warn = __reduce_or_sync(0xffffffffu, warn);
      st = __reduce_or_sync(0xffffffffu, st) | warn;
    }
    int y = -1;
    bool failed = bad_T || J < 0;
    if (!failed && !greedy) {
      const float uG = __shfl_sync(0xffffffffu, ux, P.gamma);  // meaningful in the first warp
      if (gwarp == 0 && lane == 0) gs.row.w = uG;
      group_sync(group);
      const float ud = gs.row.w;
      if (!(ud >= 0.f && ud < 1.f)) {
        st |= SPECDEC_STATUS_BAD_UNIFORM;
        failed = true;
      } else {
        const T* lrow = static_cast<const T*>(P.logits) + (static_cast<int64_t>(b) * R + J) * P.V;
        const float* qrow = (J < P.gamma) ? P.q + (static_cast<int64_t>(b) * P.gamma + J) * P.V : nullptr;
        bool zr = false, bq = false;
        y = draw_pass<T>(P, lrow, qrow, rs.m, c, 1.f / rs.Z, ud, pp, gs, group, gwarp, lane, zr, bq);
        if (bq) {
          st |= SPECDEC_STATUS_BAD_PROB;
          failed = true;
        } else if (zr) {
          st |= SPECDEC_STATUS_ZERO_RESIDUAL;
        }
      }
    } else if (!failed) {
      y = rs.z;
    }

    if (gwarp == 0) {
      const int Jo = failed ? -1 : J;
      if (lane < R) {
        int tok = -1;
        if (Jo >= 0) {
          if (lane < Jo) tok = x;
          else if (lane == Jo) tok = y;
        }
        P.out_tokens[static_cast<int64_t>(b) * R + lane] = tok;
      }
      if (lane < P.gamma && P.out_p_draft)
        P.out_p_draft[static_cast<int64_t>(b) * P.gamma + lane] = (!failed && lane <= Jo) ? px : kNaN;
      if (lane == 0) {
        P.out_J[b] = Jo;
        if (P.out_status) P.out_status[b] = failed && bad_T ? SPECDEC_STATUS_BAD_TEMPERATURE : st;
      }
    }
    group_sync(group);
  }
  // Copies still in flight after a bounded wait gave up: wait (bounded) before exiting.
  if (!pp.ok && lane == 0)
    for (; pp.k < pp.issued; ++pp.k) mbar_wait(pp.sbar(pp.k), (pp.k / kSeqStages) & 1u);
}

}  // namespace

cudaError_t launch_chain_seq(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream) {
  constexpr int smem = kSeqWarps * kSeqStages * kSeqChunkBytes;
  static unsigned long long configured_bf16 = 0, configured_f32 = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  const unsigned long long bit = 1ull << (dev & 63);
  const void* kern = (ldt == SPECDEC_BF16) ? reinterpret_cast<const void*>(chain_seq_kernel<uint16_t>)
                                           : reinterpret_cast<const void*>(chain_seq_kernel<float>);
  unsigned long long& configured = (ldt == SPECDEC_BF16) ? configured_bf16 : configured_f32;
  if (!(configured & bit)) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured |= bit;
  }
  const dim3 grid(P.grid_stats), block(kSeqWarps * 32);
  if (ldt == SPECDEC_BF16) return launch_kernel(chain_seq_kernel<uint16_t>, grid, block, smem, stream, 0, P);
  return launch_kernel(chain_seq_kernel<float>, grid, block, smem, stream, 0, P);
}

}  // namespace specdec
