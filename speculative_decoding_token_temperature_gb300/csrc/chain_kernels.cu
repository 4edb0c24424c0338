// Chain (and greedy) verification kernels.
//
// Statistics kernel: one CTA per (sequence, row, segment) computes the segment's maximum,
// its sum of 2^((l - max) * log2(e) / T) and the lowest index of the maximum in a single
// pass over the logits (16-byte coalesced loads).  The last CTA of a sequence to finish
// (an arrival counter, no waiting) merges the segments of every row and runs the accept
// tests in order: SD 20.5, "A round of speculative sampling" -- accept x_i iff
// u_i < p_i(x_i) / q_i(x_i), J = leading accepts; greedy sequences compare with the
// argmax instead ("A round of greedy speculative decoding").
//
// Draw kernel: one CTA per (sequence, segment) of the single row the extra token comes
// from computes the residual weights (p_J - q_J)+ (q == 0 for the bonus row; SD 20.5,
// "The speculative sampling rule" and "Speculative verification in PyTorch") and their
// segment mass; the last CTA of the sequence locates the segment holding u * S and scans
// it in index order for the smallest k with C_k > u * S (inverse CDF).

#include <cfloat>
#include <climits>

#include "specdec_device.cuh"
#include "specdec_internal.h"

namespace specdec {

namespace {



__device__ __forceinline__ bool is_greedy(float T) { return !(T >= SPECDEC_GREEDY_TEMPERATURE); }

template <typename T, int VEC, int NV, int NT>
__device__ void chain_decide(const ChainParams& P, int b) {
  __shared__ float s_m[kMaxGamma + 1];
  __shared__ float s_Z[kMaxGamma + 1];
  __shared__ int s_z[kMaxGamma + 1];
  __shared__ int s_err[kMaxGamma + 1];
  __shared__ int s_warn[kMaxGamma + 1];
  __shared__ unsigned char s_acc[kMaxGamma + 1];
  __shared__ float s_px[kMaxGamma + 1];
  __shared__ int s_stat, s_J;
  const int tid = threadIdx.x;
  const int R = P.gamma + 1;
  const float Tb = P.greedy_only ? 0.f : __ldg(P.temps + b);
  const bool greedy = P.greedy_only || is_greedy(Tb);
  const float c = greedy ? 0.f : kLog2e / Tb;
  constexpr float kNaN = __builtin_nanf("");

  // Merge the segment statistics of every row (fixed segment order: deterministic).
  for (int r = tid; r < R; r += NT) {
    const float4* pp = P.ws.partials + (static_cast<int64_t>(b) * R + r) * P.nseg;
    float m = -kInf;
    for (int s = 0; s < P.nseg; ++s) m = max_nan(m, __ldcg(pp + s).x);
    float Z = 0.f;
    int z = INT_MAX;
    const bool finite = (m == m) && m < kInf && m > -kInf;
    for (int s = 0; s < P.nseg; ++s) {
      const float4 f = __ldcg(pp + s);
      if (!greedy && finite && f.x > -kInf) Z += f.y * ex2((f.x - m) * c);
      if (f.x == m && z == INT_MAX) z = __float_as_int(f.z);
    }
    s_m[r] = m;
    s_Z[r] = Z;
    s_z[r] = z;
  }
  __syncthreads();

  // Every position's checks in parallel, in the order: logits row, draft token, then
  // (when sampled) draft probability and uniform together.
  for (int i = tid; i < R; i += NT) {
    const float m = s_m[i];
    int err = 0;
    if (!(m == m) || m == kInf) err = SPECDEC_STATUS_BAD_LOGIT;
    else if (m == -kInf) err = SPECDEC_STATUS_EMPTY_ROW;
    int warn = 0, acc = 0;
    float px = kNaN;
    if (!err && i < P.gamma) {
      const int x = __ldg(P.drafts + static_cast<int64_t>(b) * P.gamma + i);
      if (x < 0 || x >= P.V) {
        err = SPECDEC_STATUS_BAD_TOKEN;
      } else if (greedy) {
        acc = (x == s_z[i]);
      } else {
        const float qx = __ldg(P.q + (static_cast<int64_t>(b) * P.gamma + i) * P.V + x);
        const float uu = __ldg(P.u + static_cast<int64_t>(b) * R + i);
        if (!(qx >= 0.f && qx < kInf)) err |= SPECDEC_STATUS_BAD_PROB;
        if (!(uu >= 0.f && uu < 1.f)) err |= SPECDEC_STATUS_BAD_UNIFORM;
        if (!err) {
          const T* lrow = static_cast<const T*>(P.logits) + (static_cast<int64_t>(b) * R + i) * P.V;
          px = ex2((Elem<T>::load(lrow, x) - m) * c) / s_Z[i];
          if (qx == 0.f) {
            warn = SPECDEC_STATUS_ZERO_Q;
            acc = px > 0.f;
          } else {
            acc = uu * qx < px;
          }
        }
      }
    }
    s_err[i] = err;
    s_warn[i] = warn;
    s_acc[i] = static_cast<unsigned char>(acc);
    s_px[i] = px;
  }
  __syncthreads();

  // Left to right, stopping at the first error or rejection (SD 20.5, "A whole round of
  // speculative sampling").
  if (tid == 0) {
    int st = 0, J = P.gamma;
    for (int i = 0; i < R; ++i) {
      if (s_err[i]) {
        st |= s_err[i];
        J = -1;
        break;
      }
      st |= s_warn[i];
      if (i == P.gamma || !s_acc[i]) {
        J = i;
        break;
      }
    }
    if (!P.greedy_only && !(Tb - Tb == 0.f)) {
      st = SPECDEC_STATUS_BAD_TEMPERATURE;
      J = -1;
    }
    if (J >= 0 && !greedy) {
      const float uG = __ldg(P.u + static_cast<int64_t>(b) * R + P.gamma);
      if (!(uG >= 0.f && uG < 1.f)) {
        st |= SPECDEC_STATUS_BAD_UNIFORM;
        J = -1;
      }
    }
    s_stat = st;
    s_J = J;
  }
  __syncthreads();
  const int J = s_J;
  const int32_t* xb = P.drafts + static_cast<int64_t>(b) * P.gamma;
  int32_t* tb = P.out_tokens + static_cast<int64_t>(b) * R;
  for (int pos = tid; pos < R; pos += NT) {
    int tok = -1;
    if (J >= 0) {
      if (pos < J) tok = __ldg(xb + pos);
      else if (pos == J && greedy) tok = s_z[J];
    }
    tb[pos] = tok;
    if (P.out_p_draft && pos < P.gamma)
      P.out_p_draft[static_cast<int64_t>(b) * P.gamma + pos] = (J >= 0 && pos <= J) ? s_px[pos] : kNaN;
  }
  if (tid == 0) {
    P.out_J[b] = J;
    if (P.out_status) P.out_status[b] = s_stat;
    const bool draw = (J >= 0) && !greedy;
    SeqState st;
    st.meta = make_int4(J, draw ? 1 : 0, s_stat, 0);
    st.row = make_float4(draw ? s_m[J] : 0.f, draw ? s_Z[J] : 0.f, c,
                         draw ? __ldg(P.u + static_cast<int64_t>(b) * R + P.gamma) : 0.f);
    P.ws.seq[b] = st;
    P.ws.counters[b] = 0u;  // leave the arrival counter zeroed for the next call
  }
}

template <typename T, int VEC, int NV, int NT>
__global__ void __launch_bounds__(NT) chain_stats_kernel(const ChainParams P) {
  constexpr int SEG = NT * NV * VEC;
  __shared__ float sh_f[32];
  __shared__ int sh_i[32];
  __shared__ int s_last;
  const int R = P.gamma + 1;
  const int64_t item = blockIdx.x;
  const int s = static_cast<int>(item % P.nseg);
  const int64_t row = item / P.nseg;
  const int b = static_cast<int>(row / R);
  const T* lrow = static_cast<const T*>(P.logits) + row * P.V;
  const float Tb = P.greedy_only ? 0.f : __ldg(P.temps + b);
  const bool greedy = P.greedy_only || is_greedy(Tb);
  const float c = greedy ? 0.f : kLog2e / Tb;
  const int k0 = s * SEG;
  const int n = min(SEG, P.V - k0);

  float v[NV][VEC];
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int off = (j * NT + threadIdx.x) * VEC;
    if (off < n) {
      VecLoad<T, VEC>::load(lrow, k0 + off, v[j]);
    } else {
#pragma unroll
      for (int e = 0; e < VEC; ++e) v[j][e] = -kInf;
    }
  }

  float mt = -kInf;
#pragma unroll
  for (int j = 0; j < NV; ++j)
#pragma unroll
    for (int e = 0; e < VEC; ++e) mt = max_nan(mt, v[j][e]);
  const float m = Block<NT>::max(mt, sh_f);

  float Z = 0.f;
  if (!greedy) {
    float zt = 0.f;
    if (mt > -kInf) {
      float part[NV];
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) a += ex2((v[j][e] - mt) * c);
        part[j] = a;
      }
#pragma unroll
      for (int w = 1; w < NV; w <<= 1)
#pragma unroll
        for (int j = 0; j + w < NV; j += 2 * w) part[j] += part[j + w];
      zt = part[0] * ex2((mt - m) * c);
    }
    Z = Block<NT>::sum(zt, sh_f);
  }

  int idx = INT_MAX;
  if (mt == m) {
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int off = (j * NT + threadIdx.x) * VEC;
#pragma unroll
      for (int e = 0; e < VEC; ++e)
        if (idx == INT_MAX && off + e < n && v[j][e] == m) idx = k0 + off + e;
    }
  }
  idx = Block<NT>::min_int(idx, sh_i);

  if (threadIdx.x == 0) {
    P.ws.partials[item] = make_float4(m, Z, __int_as_float(idx), 0.f);
    __threadfence();
    const unsigned prev = atomicAdd(P.ws.counters + b, 1u);
    s_last = (prev == static_cast<unsigned>(R * P.nseg - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  chain_decide<T, VEC, NV, NT>(P, b);
}

// Residual (or target) weights of VEC consecutive elements and their fp32 running sum in
// index order; the same function serves the segment masses and the final scan, so the
// two agree bit for bit on every vector.
template <typename T, int VEC>
__device__ __forceinline__ float draw_weights(const T* lrow, const float* qrow, int64_t k,
                                              float c, float m, float invZ, bool use_p,
                                              float (&w)[VEC], float& psum, bool& bad_q) {
  float l[VEC];
  VecLoad<T, VEC>::load(lrow, k, l);
  float qv[VEC];
  if (qrow != nullptr && !use_p) {
    load_q<VEC>(qrow, k, qv);
  } else {
#pragma unroll
    for (int e = 0; e < VEC; ++e) qv[e] = 0.f;
  }
  float acc = 0.f, pacc = 0.f;
#pragma unroll
  for (int e = 0; e < VEC; ++e) {
    bad_q |= !(qv[e] >= 0.f && qv[e] < kInf);
    const float p = ex2((l[e] - m) * c) * invZ;
    w[e] = fmaxf(p - qv[e], 0.f);
    acc += w[e];
    pacc += p;
  }
  psum = pacc;
  return acc;
}

template <typename T, int VEC, int NV, int NT>
__device__ void chain_draw_finish(const ChainParams& P, int b, const SeqState& st) {
  constexpr int SEG = NT * NV * VEC;
  __shared__ double sh_d[32];
  __shared__ int sh_i[32];
  __shared__ int s_seg, s_usep, s_y;
  __shared__ double s_base, s_target;
  const int tid = threadIdx.x;
  const int R = P.gamma + 1;
  const int J = st.meta.x;
  const double2* dp = P.ws.draw + static_cast<int64_t>(b) * P.nseg;

  __shared__ int s_bad;
  if (tid == 0) {
    double S = 0.0;
    for (int s = 0; s < P.nseg; ++s) S += __ldcg(dp + s).x;
    s_bad = (S != S);
    const int use_p = !(S > 0.0);
    if (use_p) {
      S = 0.0;
      for (int s = 0; s < P.nseg; ++s) S += __ldcg(dp + s).y;
    }
    const double target = static_cast<double>(st.row.w) * S;
    double acc = 0.0, base_last = 0.0;
    int seg = -1, last_pos = 0;
    for (int s = 0; s < P.nseg; ++s) {
      const double2 d = __ldcg(dp + s);
      const double w = use_p ? d.y : d.x;
      if (w > 0.0) { last_pos = s; base_last = acc; }
      if (seg < 0 && acc + w > target) { seg = s; s_base = acc; }
      acc += w;
    }
    if (seg < 0) { seg = last_pos; s_base = base_last; }
    s_seg = seg;
    s_usep = use_p;
    s_target = target;
    s_y = -1;
  }
  __syncthreads();
  if (s_bad) {
    // SPECDEC_STATUS_BAD_PROB: the sequence's outputs become -1
    for (int pos = tid; pos < R; pos += NT) P.out_tokens[static_cast<int64_t>(b) * R + pos] = -1;
    if (tid == 0) {
      P.out_J[b] = -1;
      if (P.out_status) P.out_status[b] = st.meta.z | SPECDEC_STATUS_BAD_PROB;
      P.ws.counters[P.B + b] = 0u;
    }
    return;
  }
  const int seg = s_seg;
  const bool use_p = s_usep != 0;
  const double target = s_target;
  double base = s_base;

  const T* lrow = static_cast<const T*>(P.logits) + (static_cast<int64_t>(b) * R + J) * P.V;
  const float* qrow = (J < P.gamma) ? P.q + (static_cast<int64_t>(b) * P.gamma + J) * P.V : nullptr;
  const float c = st.row.z, mrow = st.row.x, invZ = 1.f / st.row.y;
  const int k0 = seg * SEG;
  const int n = min(SEG, P.V - k0);
  int last_positive = -1;
  for (int t = 0; t < NV; ++t) {
    const int off = (t * NT + tid) * VEC;
    float w[VEC];
    float vs = 0.f, ps = 0.f;
    if (off < n) {
      // with use_p the weights are p itself (the zero-residual fallback)
      bool bad_q = false;
      vs = draw_weights<T, VEC>(lrow, qrow, k0 + off, c, mrow, invZ, use_p, w, ps, bad_q);
#pragma unroll
      for (int e = 0; e < VEC; ++e)
        if (w[e] > 0.f) last_positive = k0 + off + e;
    } else {
#pragma unroll
      for (int e = 0; e < VEC; ++e) w[e] = 0.f;
    }
    double total;
    const double incl = Block<NT>::inclusive_scan(static_cast<double>(vs), sh_d, total);
    if (base + total > target) {
      const int cand = (base + incl > target) ? tid : INT_MAX;
      const int first = Block<NT>::min_int(cand, sh_i);
      if (tid == first) {
        const double excl = base + (incl - static_cast<double>(vs));
        float run = 0.f;
        int y = -1, lastp = -1;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          run += w[e];
          if (w[e] > 0.f) lastp = k0 + off + e;
          if (y < 0 && excl + static_cast<double>(run) > target) y = k0 + off + e;
        }
        s_y = (y >= 0) ? y : lastp;
      }
      __syncthreads();
      break;
    }
    base += total;
  }
  __syncthreads();
  int y = s_y;
  if (y < 0) {
    // Rounding left u * S at or past the end: take the last positive weight of the segment.
    int lp = last_positive;
    lp = -Block<NT>::min_int(lp < 0 ? INT_MAX : -lp, sh_i);
    y = lp;
  }
  if (tid == 0) {
    P.out_tokens[static_cast<int64_t>(b) * R + J] = y;
    if (use_p && P.out_status) P.out_status[b] = st.meta.z | SPECDEC_STATUS_ZERO_RESIDUAL;
    P.ws.counters[P.B + b] = 0u;
  }
}

template <typename T, int VEC, int NV, int NT>
__global__ void __launch_bounds__(NT) chain_sample_kernel(const ChainParams P) {
  constexpr int SEG = NT * NV * VEC;
  __shared__ double sh_d[32];
  __shared__ int s_last;
  const int s = blockIdx.x;
  const int b = blockIdx.y;
  SeqState st;
  st.meta = __ldcg(&P.ws.seq[b].meta);
  if (st.meta.y == 0) return;
  st.row = __ldcg(&P.ws.seq[b].row);
  const int R = P.gamma + 1;
  const int J = st.meta.x;
  const T* lrow = static_cast<const T*>(P.logits) + (static_cast<int64_t>(b) * R + J) * P.V;
  const float* qrow = (J < P.gamma) ? P.q + (static_cast<int64_t>(b) * P.gamma + J) * P.V : nullptr;
  const float c = st.row.z, mrow = st.row.x, invZ = 1.f / st.row.y;
  const int k0 = s * SEG;
  const int n = min(SEG, P.V - k0);

  double sr = 0.0, sp = 0.0;
  bool bad_q = false;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int off = (j * NT + threadIdx.x) * VEC;
    if (off < n) {
      float w[VEC], ps;
      sr += static_cast<double>(draw_weights<T, VEC>(lrow, qrow, k0 + off, c, mrow, invZ, false, w, ps, bad_q));
      sp += static_cast<double>(ps);
    }
  }
  // a NaN, infinite or negative draft probability in the drawn row poisons the mass
  if (bad_q) sr = __longlong_as_double(0x7ff8000000000000LL);
  sr = Block<NT>::sum(sr, sh_d);
  sp = Block<NT>::sum(sp, sh_d);
  if (threadIdx.x == 0) {
    P.ws.draw[static_cast<int64_t>(b) * P.nseg + s] = make_double2(sr, sp);
    __threadfence();
    const unsigned prev = atomicAdd(P.ws.counters + P.B + b, 1u);
    s_last = (prev == static_cast<unsigned>(P.nseg - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  chain_draw_finish<T, VEC, NV, NT>(P, b, st);
}

template <typename T, int VEC, int NV>
cudaError_t launch_stats_t(const ChainParams& P, cudaStream_t stream) {
  const int64_t items = static_cast<int64_t>(P.B) * (P.gamma + 1) * P.nseg;
  return launch_kernel(chain_stats_kernel<T, VEC, NV, kChainThreads>, dim3(static_cast<unsigned>(items)),
                       dim3(kChainThreads), 0, stream, 0, P);
}

template <typename T, int VEC, int NV>
cudaError_t launch_sample_t(const ChainParams& P, cudaStream_t stream) {
  return launch_kernel(chain_sample_kernel<T, VEC, NV, kChainThreads>, dim3(P.nseg, P.B),
                       dim3(kChainThreads), 0, stream, 0, P);
}

}  // namespace

int chain_segment_len(specdec_dtype ldt, bool vector_path) {
  if (!vector_path) return kChainThreads * kScalarElemsPerThread;
  return kChainThreads * kChainVectorsPerThread * (ldt == SPECDEC_BF16 ? 8 : 4);
}

cudaError_t launch_chain_stats(const ChainParams& P, specdec_dtype ldt, bool vector_path,
                               cudaStream_t stream) {
  if (vector_path) {
    if (ldt == SPECDEC_BF16) return launch_stats_t<uint16_t, 8, kChainVectorsPerThread>(P, stream);
    return launch_stats_t<float, 4, kChainVectorsPerThread>(P, stream);
  }
  if (ldt == SPECDEC_BF16) return launch_stats_t<uint16_t, 1, kScalarElemsPerThread>(P, stream);
  return launch_stats_t<float, 1, kScalarElemsPerThread>(P, stream);
}

cudaError_t launch_chain_sample(const ChainParams& P, specdec_dtype ldt, bool vector_path,
                                cudaStream_t stream) {
  if (vector_path) {
    if (ldt == SPECDEC_BF16) return launch_sample_t<uint16_t, 8, kChainVectorsPerThread>(P, stream);
    return launch_sample_t<float, 4, kChainVectorsPerThread>(P, stream);
  }
  if (ldt == SPECDEC_BF16) return launch_sample_t<uint16_t, 1, kScalarElemsPerThread>(P, stream);
  return launch_sample_t<float, 1, kScalarElemsPerThread>(P, stream);
}

}  // namespace specdec
