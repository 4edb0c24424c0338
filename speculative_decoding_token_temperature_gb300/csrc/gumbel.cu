// Gumbel-coupled verification and the drafter's shared-noise sampler.
//
// Art of Guessing, "Gumbel coupling" (Daliri et al.): the drafter and the target use the
// same noise g_k at draft position k.  The drafter proposes x_k = argmax_i (log q_k(i) + g_k,i);
// the target samples t_k = argmax_i (log p_k(i) + g_k,i); the round keeps the drafts while
// x_k == t_k and emits t_k at the first position where they differ.
// Verification is exact matching, and the emitted text is what the target alone samples
// with that noise, whatever the drafter.
//
// The noise never touches memory: every thread regenerates it with Philox4x32-10 (Salmon,
// Moraes, Dror, Shaw, SC 2011), written from that definition.  Entries 4j..4j+3 of row k
// of sequence b take the four outputs of counter (j, k, b, 0) under key (seed low, seed
// high); an output x gives u = ((x >> 9) + 0.5) / 2^23 (exact in float32, inside (0, 1)).
// The race runs in log2 units: score_i = a_i - log2(xi_i), xi_i = -ln(u_i) computed as
// -log1p(u_i - 1) (u - 1 is exact, so xi keeps its relative accuracy where u is near 1,
// which is where the winners are), a_i = l_i * log2(e) / T for the target, log2(q_i) for
// the drafter.  Ties go to the lowest index.
//
// The noise value G = -log2(xi) is evaluated with the hardware base-2 logarithm where its
// absolute error is small against the result: t = -log2(u) directly for u <= 0.75, and for
// u > 0.75 xi = -ln(1 + x), x = u - 1, from the series ln(1 + x) = 2 atanh(y) =
// 2 (y + y^3/3 + y^5/5 + y^7/7 + y^9/9), y = x / (2 + x), |y| <= 1/7 (truncation below
// 1e-9 relative); then G = -log2(t) + log2(log2(e)) or -log2(xi).  Against the float64
// definition the error stays within two float32 ulps of G (below 4e-6, tested), far inside
// the parity rule's tie band.
//
// Entries that cannot win are skipped: u <= 1 - 2^-24 bounds G <= 24, so once some entry
// has score L, any entry with a_i + 24.25 < L is out of the race.  Each part of a row first
// finds its largest a and scores that entry (L), then races only its entries within 24.25
// of L; of those, an entry whose noise bound -log2(1 - u) (from -ln u >= 1 - u) cannot
// lift it to L is dropped before its noise is computed.
//
// verify: rows are evaluated left to right in waves of two rows of every sequence still
//         open, each row split across CTAs (parts); a decision kernel merges the parts,
//         compares with the drafts and closes the sequences whose round is decided, so
//         the rows after the first disagreement's wave are not read.  The whole GPU works
//         on every wave instead of one CTA walking each sequence.
// draft:  one CTA per (sequence, position) races the q row.

#include <algorithm>
#include <climits>

#include "specdec_device.cuh"
#include "specdec_internal.h"

namespace specdec {

namespace {

constexpr int kGumbelThreads = 512;
constexpr int kGumbelMaxParts = 16;  // CTAs per row at most

// Philox4x32-10's round keys, (k0, k1) of rounds 0..9: the key bumped by the Weyl
// constants before every round but the first.  Built on the host once per call and
// passed as a kernel parameter, so each round reads its keys from the constant bank.
struct PhiloxKeys {
  uint32_t k[20];
};
PhiloxKeys philox_keys(uint64_t seed) {
  PhiloxKeys ks;
  uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    ks.k[2 * r] = k0;
    ks.k[2 * r + 1] = k1;
  }
  return ks;
}

// One Philox4x32-10 block (Salmon et al., SC 2011): ten rounds of two 32x32 -> 64-bit
// products, their halves crossed with the other two words and the round keys.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxKeys& ks) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * c.x;
    const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * c.z;
    c = make_uint4(static_cast<uint32_t>(p1 >> 32) ^ c.y ^ ks.k[2 * r], static_cast<uint32_t>(p1),
                   static_cast<uint32_t>(p0 >> 32) ^ c.w ^ ks.k[2 * r + 1], static_cast<uint32_t>(p0));
  }
  return c;
}

// u = ((x >> 9) + 1/2) 2^-23, built from the bits: 1 + (x >> 9) 2^-23 is the float with
// those 23 mantissa bits, and subtracting 1 - 2^-24 from it is exact (Sterbenz).
__device__ __forceinline__ float uniform_of(uint32_t x) {
  return __fsub_rn(__uint_as_float(0x3F800000u | (x >> 9)), 0.99999994039535522f);
}

constexpr float kLog2Log2e = 0.52876637294489777f;  // log2(log2(e))
constexpr float kNoiseMax = 24.25f;                  // above every G (u <= 1 - 2^-24)

__device__ __forceinline__ float lg2_approx(float x) {
  float r;
  asm("lg2.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// G = -log2(xi), xi = -ln(u)
__device__ __forceinline__ float neg_log2_xi(float u) {
  if (u <= 0.75f) return kLog2Log2e - lg2_approx(-lg2_approx(u));  // -log2(-log2(u) ln 2)
  const float x = u - 1.f;                                         // exact
  const float y = __fdividef(x, 2.f + x);
  const float y2 = y * y;
  const float s = fmaf(y2, fmaf(y2, fmaf(y2, fmaf(y2, 1.f / 9.f, 1.f / 7.f), 1.f / 5.f), 1.f / 3.f), 1.f);
  return -lg2_approx(-2.f * y * s);                                // xi = -ln(1 + x) = -2 atanh(y)
}

// Since -ln u >= 1 - u, G = -log2(-ln u) <= -log2(1 - u) (1 - u is exact in float32).  An
// entry whose a - log2(1 - u) stays below the top entry's score s_top cannot win or tie:
// one base-2 logarithm rejects most entries before the noise itself is computed.  The
// slack covers lg2.approx's error and that of the computed G (below 4e-6).
constexpr float kBoundSlack = 1e-3f;
__device__ __forceinline__ bool cannot_reach(float a, float u, float s_top) {
  return a - lg2_approx(1.f - u) + kBoundSlack < s_top;
}

struct Best {
  float s;
  int i;
};
__device__ __forceinline__ void take(Best& b, float s, int i) {  // entries arrive in index order
  if (s > b.s) {
    b.s = s;
    b.i = i;
  }
}
__device__ __forceinline__ Best better(const Best& a, const Best& b) {
  if (a.s > b.s) return a;
  if (b.s > a.s) return b;
  return a.i <= b.i ? a : b;
}

// Block-wide (best score, lowest index) and the NaN-propagating maximum logit.
template <int NT>
__device__ __forceinline__ void block_best(Best& b, float& mx, Best* sh_b, float* sh_m) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Best t;
    t.s = __shfl_xor_sync(0xffffffffu, b.s, o);
    t.i = __shfl_xor_sync(0xffffffffu, b.i, o);
    b = better(b, t);
    mx = max_nan(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  __syncthreads();
  if (l == 0) {
    sh_b[w] = b;
    sh_m[w] = mx;
  }
  __syncthreads();
  b = sh_b[0];
  mx = sh_m[0];
#pragma unroll
  for (int i = 1; i < NT / 32; ++i) {
    b = better(b, sh_b[i]);
    mx = max_nan(mx, sh_m[i]);
  }
}

// Every group of 4 entries of a row, in index order per thread: thread t takes 16-byte
// vectors t, t + NT, ... (2 groups per bf16 vector, 1 per fp32 vector), kUnroll vectors
// loaded before any is used, so that many loads are in flight; f(j, v) gets group j's four
// values (-inf past V).  VEC needs rows of whole, 16-byte aligned vectors; other rows are
// read entry by entry.
constexpr int kUnroll = 4;
template <typename T, bool VEC, int NT, typename F>
__device__ __forceinline__ void for_groups(const T* row, int V, int part, int parts, F&& f) {
  const int ng = (V + 3) / 4;
  if constexpr (VEC) {
    constexpr int GPV = 16 / (4 * static_cast<int>(sizeof(T)));  // groups per 16-byte vector
    const int nv = (ng + GPV - 1) / GPV;
    const int va = static_cast<int>(static_cast<int64_t>(nv) * part / parts);
    const int vb = static_cast<int>(static_cast<int64_t>(nv) * (part + 1) / parts);
    for (int v0 = va + threadIdx.x; v0 < vb; v0 += kUnroll * NT) {
      uint4 w[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int vi = v0 + u * NT;
        if (vi < vb) w[u] = __ldg(reinterpret_cast<const uint4*>(row) + vi);  // rows hold whole vectors
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int vi = v0 + u * NT;
        if (vi >= vb) break;
#pragma unroll
        for (int g = 0; g < GPV; ++g) {
          const int j = vi * GPV + g;
          if (j >= ng) break;
          float v[4];
          if constexpr (sizeof(T) == 2) {
            const uint32_t a = g ? w[u].z : w[u].x, c = g ? w[u].w : w[u].y;
            v[0] = bf16_lo(a); v[1] = bf16_hi(a); v[2] = bf16_lo(c); v[3] = bf16_hi(c);
          } else {
            v[0] = __uint_as_float(w[u].x); v[1] = __uint_as_float(w[u].y);
            v[2] = __uint_as_float(w[u].z); v[3] = __uint_as_float(w[u].w);
          }
          f(j, v);
        }
      }
    }
  } else {
    const int ga = static_cast<int>(static_cast<int64_t>(ng) * part / parts);
    const int gb = static_cast<int>(static_cast<int64_t>(ng) * (part + 1) / parts);
    for (int j0 = ga + threadIdx.x; j0 < gb; j0 += kUnroll * NT) {
      float v[kUnroll][4];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int j = j0 + u * NT;
#pragma unroll
        for (int e = 0; e < 4; ++e) v[u][e] = (j < gb && 4 * j + e < V) ? Elem<T>::load(row, 4 * j + e) : -kInf;
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (j0 + u * NT < gb) f(j0 + u * NT, v[u]);
    }
  }
}

// One part of one row's race (a CTA): the part's largest logit and its lowest index, then
// the race over the part's entries within kNoiseMax of the part's own top score (an entry
// below that cannot win the part, so it cannot win the row).  Greedy: the top entry only.
struct Partial {
  float best;  // best score (greedy: the largest logit)
  int idx;     // its lowest index
  float mx;    // the largest logit (NaN if any logit is NaN)
  int pad;
};

template <typename T, bool VEC>
__device__ Partial race_part(const T* row, int V, int part, int parts, bool greedy, float c, uint32_t k, uint32_t b,
                             const PhiloxKeys& ks, Best* sh_b, float* sh_m) {
  Best top;
  top.s = -kInf;
  top.i = INT_MAX;
  float mx = -kInf;
  // the part's largest logit by group (entries past V are -inf): the group of the first
  // strict maximum, then its lowest entry holding it
  for_groups<T, VEC, kGumbelThreads>(row, V, part, parts, [&](int j, const float (&v)[4]) {
    mx = max_nan(mx, max_nan(max_nan(v[0], v[1]), max_nan(v[2], v[3])));
    take(top, fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])), j);
  });
  if (top.i != INT_MAX) {
    const int j = top.i;
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = 4 * j + e < V ? Elem<T>::load(row, 4 * j + e) : -kInf;
    int e = 0;
    while (e < 3 && !(v[e] == top.s)) ++e;
    top.i = 4 * j + e;
  }
  block_best<kGumbelThreads>(top, mx, sh_b, sh_m);
  Partial out;
  out.mx = mx;
  out.pad = 0;
  if (greedy || top.i == INT_MAX || !(mx == mx) || mx == kInf) {
    out.best = top.s;
    out.idx = top.i;
    return out;
  }
  const int jt = top.i >> 2;
  const uint4 xt = philox4x32_10(make_uint4(static_cast<uint32_t>(jt), k, b, 0u), ks);
  const uint32_t xts[4] = {xt.x, xt.y, xt.z, xt.w};
  const float score_top = __fsub_rn(__fmul_rn(top.s, c), -neg_log2_xi(uniform_of(xts[top.i & 3])));
  const float cut = score_top - kNoiseMax;
  Best best;
  best.s = -kInf;
  best.i = INT_MAX;
  float unused = -kInf;
  for_groups<T, VEC, kGumbelThreads>(row, V, part, parts, [&](int j, const float (&v)[4]) {
    float a[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) a[e] = (4 * j + e < V) ? __fmul_rn(v[e], c) : -kInf;
    if (fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3])) < cut) return;
    const uint4 x = philox4x32_10(make_uint4(static_cast<uint32_t>(j), k, b, 0u), ks);
    const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (!(a[e] >= cut)) continue;
      const float u = uniform_of(xs[e]);
      if (cannot_reach(a[e], u, score_top)) continue;
      take(best, __fsub_rn(a[e], -neg_log2_xi(u)), 4 * j + e);
    }
  });
  block_best<kGumbelThreads>(best, unused, sh_b, sh_m);
  out.best = best.s;
  out.idx = best.i;
  return out;
}

// Rows are evaluated in waves of kWaveRows rows of every sequence still open: one CTA per
// (sequence, row of the wave, part of the row), then one decision per sequence.
constexpr int kWaveRows = 2;

__device__ __forceinline__ const Partial* partials_of(const GumbelParams& P, int b, int r) {
  return reinterpret_cast<const Partial*>(P.partials) + (static_cast<int64_t>(b) * kWaveRows + r) * P.parts;
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(kGumbelThreads, 2) gumbel_wave_kernel(const GumbelParams P, int wave,
                                                                     const __grid_constant__ PhiloxKeys ks) {
  __shared__ Best sh_b[kGumbelThreads / 32];
  __shared__ float sh_m[kGumbelThreads / 32];
  const int part = blockIdx.x % P.parts;
  const int r = (blockIdx.x / P.parts) % kWaveRows;
  const int b = blockIdx.x / (P.parts * kWaveRows);
  const int k = wave * kWaveRows + r;
  // Launched early behind the previous decision (programmatic dependent launch): let the
  // next kernel start early too, then wait for the decisions this wave reads.
  grid_launch_dependents();
  grid_dependency_wait();
  if (k > P.G || __ldcg(P.state + b) != 0) return;  // past the last row, or the round is decided
  const float Tb = __ldg(P.temps + b);
  const bool greedy = !(Tb >= SPECDEC_GREEDY_TEMPERATURE);
  const float c = greedy ? 1.f : kLog2e / Tb;
  const T* row = static_cast<const T*>(P.logits) + (static_cast<int64_t>(b) * (P.G + 1) + k) * P.V;
  const Partial out = race_part<T, VEC>(row, P.V, part, P.parts, greedy, c, static_cast<uint32_t>(k),
                                        static_cast<uint32_t>(b), ks, sh_b, sh_m);
  if (threadIdx.x == 0)
    reinterpret_cast<Partial*>(P.partials)[(static_cast<int64_t>(b) * kWaveRows + r) * P.parts + part] = out;
}

// One thread per sequence: merge the parts of the wave's rows in order and decide.
__global__ void __launch_bounds__(128) gumbel_decide_kernel(const GumbelParams P, int wave) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  grid_launch_dependents();
  grid_dependency_wait();  // the wave's parts
  if (b >= P.B || P.state[b] != 0) return;
  const int R = P.G + 1;
  const float Tb = __ldg(P.temps + b);
  int st = (Tb - Tb == 0.f) ? 0 : SPECDEC_STATUS_BAD_TEMPERATURE;
  int J = -1, last = -1;
  for (int r = 0; r < kWaveRows && !st && J < 0; ++r) {
    const int k = wave * kWaveRows + r;
    if (k > P.G) break;
    const Partial* pp = partials_of(P, b, r);
    Best best;
    best.s = -kInf;
    best.i = INT_MAX;
    float mx = -kInf;
    for (int q = 0; q < P.parts; ++q) {
      const Partial x = pp[q];
      mx = max_nan(mx, x.mx);
      Best t;
      t.s = x.best;
      t.i = x.idx;
      best = better(best, t);
    }
    if (!(mx == mx) || mx == kInf) {
      st = SPECDEC_STATUS_BAD_LOGIT;
      break;
    }
    if (mx == -kInf) {
      st = SPECDEC_STATUS_EMPTY_ROW;
      break;
    }
    int x = -1;
    if (k < P.G) {
      x = __ldg(P.drafts + static_cast<int64_t>(b) * P.G + k);
      if (x < 0 || x >= P.V) {
        st = SPECDEC_STATUS_BAD_TOKEN;
        break;
      }
    }
    if (k == P.G || x != best.i) {
      J = k;
      last = best.i;
    }
  }
  if (!st && J < 0) return;  // every row of this wave agreed: the next wave continues
  int32_t* tok = P.out_tokens + static_cast<int64_t>(b) * R;
  for (int i = 0; i < R; ++i)
    tok[i] = st ? -1 : (i < J ? __ldg(P.drafts + static_cast<int64_t>(b) * P.G + i) : (i == J ? last : -1));
  P.out_J[b] = st ? -1 : J;
  if (P.out_status) P.out_status[b] = st;
  P.state[b] = 1;
}

template <bool VEC>
__global__ void __launch_bounds__(kGumbelThreads, 2) gumbel_draft_kernel(const float* __restrict__ q,
                                                                      const __grid_constant__ PhiloxKeys ks, int G,
                                                                      int V, int32_t* __restrict__ out) {
  __shared__ Best sh_b[kGumbelThreads / 32];
  __shared__ float sh_m[kGumbelThreads / 32];
  const int row = blockIdx.x;  // b * G + k
  const int b = row / G, k = row - b * G;
  const float* qr = q + static_cast<int64_t>(row) * V;
  // the largest q (NaN and negative entries never count) and its lowest index
  Best top;
  top.s = -kInf;
  top.i = INT_MAX;
  float unused = -kInf;
  for_groups<float, VEC, kGumbelThreads>(qr, V, 0, 1, [&](int j, const float (&v)[4]) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (4 * j + e < V && v[e] > 0.f) take(top, v[e], 4 * j + e);
  });
  block_best<kGumbelThreads>(top, unused, sh_b, sh_m);
  if (top.i == INT_MAX) {  // no positive entry
    if (threadIdx.x == 0) out[row] = -1;
    return;
  }
  const int jt = top.i >> 2;
  const uint4 xt = philox4x32_10(make_uint4(static_cast<uint32_t>(jt), static_cast<uint32_t>(k),
                                            static_cast<uint32_t>(b), 0u),
                                 ks);
  const uint32_t xts[4] = {xt.x, xt.y, xt.z, xt.w};
  const float score_top = __fadd_rn(log2f(top.s), neg_log2_xi(uniform_of(xts[top.i & 3])));
  const float cut = score_top - kNoiseMax;
  Best best;
  best.s = -kInf;
  best.i = INT_MAX;
  for_groups<float, VEC, kGumbelThreads>(qr, V, 0, 1, [&](int j, const float (&v)[4]) {
    float a[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) a[e] = (4 * j + e < V && v[e] > 0.f) ? log2f(v[e]) : -kInf;
    if (fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3])) < cut) return;
    const uint4 x = philox4x32_10(make_uint4(static_cast<uint32_t>(j), static_cast<uint32_t>(k),
                                             static_cast<uint32_t>(b), 0u),
                                  ks);
    const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (!(a[e] >= cut)) continue;
      const float u = uniform_of(xs[e]);
      if (cannot_reach(a[e], u, score_top)) continue;
      take(best, __fadd_rn(a[e], neg_log2_xi(u)), 4 * j + e);
    }
  });
  block_best<kGumbelThreads>(best, unused, sh_b, sh_m);
  if (threadIdx.x == 0) out[row] = best.i;
}

// The shared noise itself: out[(b * R + k) * V + i] = G of entry i, row k, sequence b.
__global__ void __launch_bounds__(256) gumbel_noise_kernel(const __grid_constant__ PhiloxKeys ks, int B, int R,
                                                           int V, float* __restrict__ out) {
  const int ng = (V + 3) / 4;
  const int64_t total = static_cast<int64_t>(B) * R * ng;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t rowi = t / ng;
    const int j = static_cast<int>(t - rowi * ng);
    const int k = static_cast<int>(rowi % R), b = static_cast<int>(rowi / R);
    const uint4 x = philox4x32_10(make_uint4(static_cast<uint32_t>(j), static_cast<uint32_t>(k),
                                             static_cast<uint32_t>(b), 0u),
                                  ks);
    const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (4 * j + e < V) out[rowi * V + 4 * j + e] = neg_log2_xi(uniform_of(xs[e]));
  }
}

}  // namespace

cudaError_t launch_gumbel_noise(uint64_t seed, int B, int R, int V, float* out, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(B) * R * ((V + 3) / 4);
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, 152 * 8);
  return launch_kernel(gumbel_noise_kernel, dim3(static_cast<unsigned>(std::max<int64_t>(blocks, 1))), dim3(256), 0,
                       stream, 0, philox_keys(seed), B, R, V, out);
}

cudaError_t launch_gumbel_verify(const GumbelParams& P, specdec_dtype ldt, bool vec, cudaStream_t stream) {
  const int waves = (P.G + 1 + kWaveRows - 1) / kWaveRows;
  const dim3 grid(static_cast<unsigned>(P.B) * kWaveRows * static_cast<unsigned>(P.parts)), block(kGumbelThreads);
  const dim3 dgrid((P.B + 127) / 128), dblock(128);
  const PhiloxKeys ks = philox_keys(static_cast<uint64_t>(P.key0) | (static_cast<uint64_t>(P.key1) << 32));
  // Every launch after the first starts while its predecessor finishes (programmatic
  // dependent launch); each kernel waits for its predecessor's results before reading them.
  for (int w = 0; w < waves; ++w) {
    cudaError_t e;
    const int pdl = w > 0 ? 1 : 0;
    if (ldt == SPECDEC_BF16)
      e = vec ? launch_kernel(gumbel_wave_kernel<uint16_t, true>, grid, block, 0, stream, pdl, P, w, ks)
              : launch_kernel(gumbel_wave_kernel<uint16_t, false>, grid, block, 0, stream, pdl, P, w, ks);
    else
      e = vec ? launch_kernel(gumbel_wave_kernel<float, true>, grid, block, 0, stream, pdl, P, w, ks)
              : launch_kernel(gumbel_wave_kernel<float, false>, grid, block, 0, stream, pdl, P, w, ks);
    if (e != cudaSuccess) return e;
    if ((e = launch_kernel(gumbel_decide_kernel, dgrid, dblock, 0, stream, 1, P, w)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int gumbel_parts(int B) {
  // At least about four CTAs per SM in the first wave (two resident at a time), and of
  // the part counts up to twice that, the one whose last round of resident CTAs is the
  // fullest (fewest SMs idle at the end of the wave).
  const int slots = 2 * device_sm_count();
  const int rows = B * kWaveRows;
  int lo = (2 * slots + rows - 1) / rows;
  lo = lo < 1 ? 1 : (lo > kGumbelMaxParts ? kGumbelMaxParts : lo);
  const int hi = std::min(kGumbelMaxParts, 2 * lo);
  int best = lo;
  double best_fill = 0.0;
  for (int p = lo; p <= hi; ++p) {
    const int64_t ctas = static_cast<int64_t>(rows) * p;
    const int64_t rounds = (ctas + slots - 1) / slots;
    const double fill = static_cast<double>(ctas) / static_cast<double>(rounds * slots);
    if (fill > best_fill + 0.02) {
      best = p;
      best_fill = fill;
    }
  }
  return best;
}

size_t gumbel_workspace_bytes(int B) {
  const size_t state = (static_cast<size_t>(B) * sizeof(int) + 255) / 256 * 256;
  return state + static_cast<size_t>(B) * kWaveRows * kGumbelMaxParts * sizeof(Partial);
}

cudaError_t launch_gumbel_draft(const float* q, uint64_t seed, int B, int G, int V, bool vec, int32_t* out,
                                cudaStream_t stream) {
  const PhiloxKeys ks = philox_keys(seed);
  const dim3 grid(static_cast<unsigned>(B) * static_cast<unsigned>(G)), block(kGumbelThreads);
  if (vec) return launch_kernel(gumbel_draft_kernel<true>, grid, block, 0, stream, 0, q, ks, G, V, out);
  return launch_kernel(gumbel_draft_kernel<false>, grid, block, 0, stream, 0, q, ks, G, V, out);
}

}  // namespace specdec
