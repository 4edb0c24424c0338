// Block verification that reads every logits row and every q row from HBM once.
//
// Art of Guessing, "Block verification" (Sun et al.): with p_k = softmax(l_k / T) and
// q_k the drafter's distribution at position k,
//   w_0 = 1, w_{k+1} = min(1, w_k p_k(x_k) / q_k(x_k)),
//   mass_k = sum_v (w_k p_k(v) - q_k(v))+ (mass_gamma = w_gamma),
//   survival_k = mass_k / (mass_k + 1 - w_k) (1 when w_k = 1),
//   n = the longest prefix k with u[k-1] <= survival_k, and the extra token is drawn from
//   (w_n p_n - q_n)+ (q_gamma = 0).
// Row k's residual needs w_k (rows 0..k-1) and Z_k (row k itself), so the rule can walk a
// sequence row by row: the statistics of row k, then at once its residual masses, a
// second read of the row that L2 still holds.  One CTA (one per SM) walks whole sequences
// this way, so only about one row per SM is live between its two reads (152 x 256 KB at
// V = 128256, bf16) and no CTA waits on another.  q rows, read once, and the second read
// of each logits row are copied with an evict-first policy.
//
// Per row k of a sequence, in one CTA of 16 warps (warp w takes items w, w + 16, ...):
//   statistics  the row's 4 KB chunks: (max, sum of 2^((l-m)c), lowest argmax) per chunk
//               into shared memory; after a barrier every warp merges them in chunk order
//               (identical bits in every warp), and the lane holding position k forms
//               p_k(x_k) and the ratio; every warp carries the running weight w.
//   masses      (sampled sequences) the row's CH-element chunks of logits and q: the chunk
//               mass of (w_k p_k - q_k)+ into shared memory, and the q check.
// After the last row warp 0 sums each row's chunk masses in fp64 in chunk order, applies
// the checks and the survival tests, scans row n's chunk masses and then the chosen chunk
// for the inverse-CDF draw, and writes the outputs.  Each warp's bulk copies (a 3-stage
// ring) run ahead across rows and sequences, so they stream through the barriers.

#include "stream_common.cuh"

namespace specdec {

namespace {

constexpr int kW = kBlockWarps;
constexpr int kStages = kBlockStages;
constexpr int kStage = kStatsChunkBytes;  // bytes per stage: one statistics chunk or one mass chunk

template <typename T>
constexpr int mass_chunk() { return sizeof(T) == 2 ? kBlockMassChunkBf16 : kBlockMassChunkF32; }
static_assert(kBlockMassChunkBf16 * (2 + 4) <= kStage, "a bf16 mass chunk exceeds a stage");
static_assert(kBlockMassChunkF32 * (4 + 4) <= kStage, "an fp32 mass chunk exceeds a stage");

struct RowShared {
  uint64_t bar[kW][kStages];         // copy stages
  float4 slot_s[2][kBlockSlotsS];    // chunk summaries of the current row (by row parity)
  float slot_m[kBlockSlotsM];        // chunk masses of the current sequence, row-major
  int qbad;                          // a bad draft probability in the current sequence
};

__device__ __forceinline__ void cta_barrier() {
  asm volatile("bar.sync 1, %0;" ::"r"(kW * 32) : "memory");
}

// Mass of one row from its nchm chunk masses (one warp): fp64 sums of lane-contiguous
// runs, then the warp's inclusive scan; every lane gets the total.  The same order as
// find_chunk below, so both see the same running masses.
__device__ __forceinline__ double row_mass(const float* sm, int nchm, int lane) {
  const int cpl = (nchm + 31) / 32;
  const int c0 = min(lane * cpl, nchm), c1 = min(c0 + cpl, nchm);
  double mine = 0.0;
  for (int q = c0; q < c1; ++q) mine += static_cast<double>(sm[q]);
  return __shfl_sync(0xffffffffu, warp_incl_scan(mine, lane), 31);
}

// The chunk of a row (masses sm[0..nchm) in shared memory) whose running mass first
// exceeds target, else the last one with mass, and the mass before it (one warp).
__device__ void find_chunk(const float* sm, int nchm, double target, int lane, int& cstar, double& before) {
  const int cpl = (nchm + 31) / 32;
  const int c0 = min(lane * cpl, nchm), c1 = min(c0 + cpl, nchm);
  double mine = 0.0;
  for (int q = c0; q < c1; ++q) mine += static_cast<double>(sm[q]);
  const double incl = warp_incl_scan(mine, lane);
  double pre = incl - mine;
  int found = -1, lastpos = -1;
  double fb = 0.0, lb = 0.0;
  for (int q = c0; q < c1; ++q) {
    const double w = static_cast<double>(sm[q]);
    if (w > 0.0) {
      lastpos = q;
      lb = pre;
    }
    if (found < 0 && pre + w > target) {
      found = q;
      fb = pre;
    }
    pre += w;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, found >= 0);
  if (hit) {
    const int fl = __ffs(hit) - 1;
    cstar = __shfl_sync(0xffffffffu, found, fl);
    before = __shfl_sync(0xffffffffu, fb, fl);
    return;
  }
  const int best = warp_max_int(lastpos);  // rounding put target at or past the row's end
  const unsigned owner = __ballot_sync(0xffffffffu, lastpos == best && best >= 0);
  cstar = best < 0 ? 0 : best;
  before = owner ? __shfl_sync(0xffffffffu, lb, __ffs(owner) - 1) : 0.0;
}

template <typename T>
__global__ void __launch_bounds__(kW * 32, 1) block_row_kernel(const ChainParams P) {
  extern __shared__ __align__(128) unsigned char stages[];
  __shared__ RowShared sh;
  constexpr int VPL = kStatsChunkBytes / 16 / 32;
  constexpr int CH = mass_chunk<T>();
  constexpr int LB = CH * static_cast<int>(sizeof(T));  // logits bytes of a full mass chunk
  constexpr int GPL = CH / 4 / 32;                      // 4-element groups per lane per mass chunk
  using GL = typename Group<T>::L;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = P.B, G = P.gamma, R = G + 1, V = P.V;
  const int nch = P.nch, nchm = P.nchm;  // R * nchm <= kBlockSlotsM, nch <= kBlockSlotsS (host)
  const int64_t row_bytes = static_cast<int64_t>(V) * sizeof(T);
  unsigned char* buf = stages + static_cast<size_t>(warp) * kStages * kStage;
  uint64_t* bar = sh.bar[warp];

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bar[s], 1);
    mbar_fence_init();
  }
  if (threadIdx.x == 0) sh.qbad = 0;
  __syncthreads();
  const uint64_t evict_first = l2_policy_evict_first();

  auto skip_of = [&](int b) {  // no mass phase: greedy or non-finite temperature
    const float Tb = __ldg(P.temps + b);
    return is_greedy(Tb) || !(Tb - Tb == 0.f);
  };
  // the copy cursor: sequence cb (this CTA's ci-th), row ck, phase cph (0 statistics,
  // 1 masses), this warp's item cj of that phase
  int ci = 0, ck = 0, cph = 0, cj = warp, cb = blockIdx.x;
  bool cskip = cb < B ? skip_of(cb) : true;
  auto normalize = [&]() {
    while (cb < B) {
      const int cnt = cph == 0 ? nch : (cskip ? 0 : nchm);
      if (cj < cnt) return;
      cj = warp;
      if (cph == 0) {
        cph = 1;
      } else {
        cph = 0;
        if (++ck == R) {
          ck = 0;
          ++ci;
          cb = blockIdx.x + ci * gridDim.x;
          if (cb < B) cskip = skip_of(cb);
        }
      }
    }
  };
  auto issue = [&](int s) {  // lane 0: the cursor's copies into stage s
    unsigned char* dst = buf + s * kStage;
    if (cph == 0) {
      const int64_t off = static_cast<int64_t>(cj) * kStatsChunkBytes;
      const uint32_t bytes = static_cast<uint32_t>(min(static_cast<int64_t>(kStatsChunkBytes), row_bytes - off));
      mbar_expect_tx(&bar[s], bytes);
      bulk_copy_g2s(dst, static_cast<const char*>(P.logits) + (static_cast<int64_t>(cb) * R + ck) * row_bytes + off,
                    bytes, &bar[s]);
    } else {
      const int n = min(CH, V - cj * CH);
      const uint32_t lb = static_cast<uint32_t>(n) * sizeof(T);
      const uint32_t qb = (ck < G) ? static_cast<uint32_t>(n) * 4u : 0u;
      const int64_t e0 = static_cast<int64_t>(cj) * CH;
      mbar_expect_tx(&bar[s], lb + qb);
      bulk_copy_g2s_hint(dst, static_cast<const T*>(P.logits) + (static_cast<int64_t>(cb) * R + ck) * V + e0, lb,
                         &bar[s], evict_first);
      if (qb)
        bulk_copy_g2s_hint(dst + LB, P.q + (static_cast<int64_t>(cb) * G + ck) * V + e0, qb, &bar[s], evict_first);
    }
  };
  normalize();
  uint32_t issued = 0, kq = 0, landed = 0;
  for (; issued < kStages && cb < B; ++issued) {
    if (lane == 0) issue(static_cast<int>(issued));
    cj += kW;
    normalize();
  }
  bool ok = true;  // false once a bounded wait gave up: the warp then only keeps the barriers
  auto wait_stage = [&]() -> int {
    const int s = static_cast<int>(kq % kStages);
    if (ok) {
      if (mbar_wait(&bar[s], (kq / kStages) & 1u)) {
        ++landed;
      } else {
        ok = false;
        if (lane == 0) atomicOr(P.ws.error, 1u);
      }
    }
    return s;
  };
  auto refill = [&](int s) {
    __syncwarp();
    ++kq;
    if (ok && cb < B) {
      if (lane == 0) {
        fence_proxy_async_smem();
        issue(s);
      }
      ++issued;
      cj += kW;
      normalize();
    }
  };

  uint32_t rows_done = 0;  // selects the summary buffer of each row
  for (int b = blockIdx.x; b < B; b += gridDim.x) {
    const float Tb = __ldg(P.temps + b);
    const bool greedy = is_greedy(Tb);
    const bool bad_T = !(Tb - Tb == 0.f);
    const bool skip = greedy || bad_T;
    const float c = greedy ? 0.f : kLog2e / Tb;

    // position inputs (lane k: position k; lane gamma: the draw's uniform)
    int x = -1, tok_err = 0, u_err = 0;
    float lx = 0.f, qx = 0.f, ux = 0.f;
    if (lane < G) {
      x = __ldg(P.drafts + static_cast<int64_t>(b) * G + lane);
      if (x < 0 || x >= V) {
        tok_err = SPECDEC_STATUS_BAD_TOKEN;
      } else if (!greedy) {
        lx = Elem<T>::load(static_cast<const T*>(P.logits) + (static_cast<int64_t>(b) * R + lane) * V, x);
        qx = __ldg(P.q + (static_cast<int64_t>(b) * G + lane) * V + x);
      }
    }
    if (!greedy && lane < R) {
      ux = __ldg(P.u + static_cast<int64_t>(b) * R + lane);
      if (!(ux >= 0.f && ux < 1.f)) u_err = SPECDEC_STATUS_BAD_UNIFORM;
    }

    // lane k ends with row k's (m, Z, argmax), p_k(x_k), w_k and w_k / Z_k
    float m_l = -kInf, Z_l = 0.f, px_l = kNaN, w_l = 1.f, a_l = 0.f;
    int z_l = INT_MAX, warn = 0;
    float w = 1.f;  // the running weight w_k, the same in every warp
    for (int k = 0; k < R; ++k) {
      float4* ss = sh.slot_s[rows_done & 1u];
      ++rows_done;
      // ---- statistics of row k
      for (int j = warp; j < nch; j += kW) {
        const int s = wait_stage();
        const int nv = static_cast<int>(min(static_cast<int64_t>(kStatsChunkBytes),
                                            row_bytes - static_cast<int64_t>(j) * kStatsChunkBytes) / 16);
        const uint4* vb = reinterpret_cast<const uint4*>(buf + s * kStage);
        uint4 v4[VPL];
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
          const int e = lane + 32 * v;
          if (e < nv) {
            v4[v] = vb[e];
          } else if constexpr (sizeof(T) == 2) {
            v4[v] = make_uint4(kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2);
          } else {
            const uint32_t ni = __float_as_uint(-kInf);
            v4[v] = make_uint4(ni, ni, ni, ni);
          }
        }
        refill(s);
        const float4 sum = chunk_summary<T>(v4, nv, static_cast<uint32_t>(j), greedy, c);
        if (lane == 0) ss[j] = sum;
      }
      cta_barrier();
      RowSum acc;  // every warp merges the row's chunks in chunk order
      acc.m = -kInf;
      acc.Z = 0.f;
      acc.z = INT_MAX;
      for (int q = lane; q < nch; q += 32) {
        const float4 f = ss[q];
        RowSum t;
        t.m = f.x;
        t.Z = f.y;
        t.z = __float_as_int(f.z);
        acc = merge(acc, t, c);
      }
      acc = warp_merge(acc, c);
      if (lane == k) {
        m_l = acc.m;
        Z_l = acc.Z;
        z_l = acc.z;
        w_l = w;
      }
      if (skip) continue;
      const float alpha = w / acc.Z;
      if (lane == k) a_l = alpha;
      if (k < G) {  // p_k(x_k), its ratio to q_k(x_k), and w_{k+1}
        float ratio = 0.f;
        if (lane == k && !tok_err) {
          px_l = ex2((lx - acc.m) * c) / acc.Z;
          if (qx == 0.f) {
            warn = SPECDEC_STATUS_ZERO_Q;
            ratio = px_l > 0.f ? kInf : 0.f;
          } else {
            ratio = px_l / qx;
          }
        }
        const float rk = __shfl_sync(0xffffffffu, ratio, k);
        w = (w == 0.f) ? 0.f : fminf(1.f, w * rk);
      }
      // ---- masses of row k
      const bool has_q = k < G;
      bool qbad_w = false;
      for (int j = warp; j < nchm; j += kW) {
        const int s = wait_stage();
        const int ng = min(CH, V - j * CH) / 4;
        const unsigned char* sb = buf + s * kStage;
        GL lw[GPL];
        float4 qv[GPL];
#pragma unroll
        for (int g = 0; g < GPL; ++g) {
          const int e = lane + 32 * g;
          if (e < ng) {
            lw[g] = reinterpret_cast<const GL*>(sb)[e];
            qv[g] = has_q ? reinterpret_cast<const float4*>(sb + LB)[e] : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        refill(s);
        float sr = 0.f;
        QCheck qc;
#pragma unroll
        for (int g = 0; g < GPL; ++g) {
          if (lane + 32 * g < ng) {
            float wv[4];
            sr += group_weights<T>(lw[g], qv[g], acc.m, c, alpha, !has_q, wv);
            qc.add(qv[g]);
          }
        }
        sr = warp_sum(sr);
        const bool bad = __any_sync(0xffffffffu, qc.bad());
        qbad_w |= bad;
        if (lane == 0) sh.slot_m[k * nchm + j] = bad ? kNaN : sr;
      }
      if (qbad_w && lane == 0) atomicOr(&sh.qbad, 1);
    }

    // ---- the decision (warp 0)
    int row_err = 0;
    if (lane < R) {
      if (!(m_l == m_l) || m_l == kInf) row_err = SPECDEC_STATUS_BAD_LOGIT;
      else if (m_l == -kInf) row_err = SPECDEC_STATUS_EMPTY_ROW;
    }
    int err = __reduce_or_sync(0xffffffffu, row_err | tok_err | u_err);
    if (bad_T) err = SPECDEC_STATUS_BAD_TEMPERATURE;
    int32_t* tok_out = P.out_tokens + static_cast<int64_t>(b) * R;
    float* pd_out = P.out_p_draft ? P.out_p_draft + static_cast<int64_t>(b) * G : nullptr;
    if (skip) {  // greedy matching (a one-hot target reduces the rule to it)
      if (warp == 0) {
        const bool miss = lane < G && x != z_l;
        const unsigned mm = __ballot_sync(0xffffffffu, miss);
        const int J = err ? -1 : (mm ? __ffs(mm) - 1 : G);
        const int zJ = __shfl_sync(0xffffffffu, z_l, J < 0 ? 0 : J);
        if (lane < R) tok_out[lane] = (J < 0) ? -1 : (lane < J ? x : (lane == J ? zJ : -1));
        if (lane < G && pd_out) pd_out[lane] = kNaN;
        if (lane == 0) {
          P.out_J[b] = J;
          if (P.out_status) P.out_status[b] = err;
        }
      }
      continue;
    }
    cta_barrier();  // every chunk mass and q check of the sequence is in shared memory
    if (warp != 0) continue;
    warn = __reduce_or_sync(0xffffffffu, warn);
    const bool qbad = sh.qbad != 0;
    __syncwarp();
    if (lane == 0) sh.qbad = 0;
    const int status = err | warn | (qbad ? SPECDEC_STATUS_BAD_PROB : 0);
    if (status & SPECDEC_STATUS_ERROR_MASK) {  // errors only: warnings describe a clean round
      if (lane < R) tok_out[lane] = -1;
      if (lane < G && pd_out) pd_out[lane] = kNaN;
      if (lane == 0) {
        P.out_J[b] = -1;
        if (P.out_status) P.out_status[b] = status & SPECDEC_STATUS_ERROR_MASK;
      }
      continue;
    }
    // survival of every prefix (mass_gamma = w_gamma) and the longest surviving one
    const float u_prev = __shfl_up_sync(0xffffffffu, ux, 1);  // lane k: u[k - 1]
    double mass_l = 0.0;
    for (int k = 1; k < G; ++k) {
      const double mk = row_mass(sh.slot_m + k * nchm, nchm, lane);
      if (lane == k) mass_l = mk;
    }
    bool survived = false;
    if (lane >= 1 && lane < R) {
      const double wk = static_cast<double>(w_l);
      const double mk = lane == G ? wk : mass_l;
      const double surv = (wk < 1.0) ? mk / (mk + 1.0 - wk) : 1.0;
      survived = static_cast<double>(u_prev) <= surv;
    }
    const unsigned sv = __ballot_sync(0xffffffffu, survived);
    const int n = sv ? 31 - __clz(sv) : 0;
    const float mN = __shfl_sync(0xffffffffu, m_l, n), zN = __shfl_sync(0xffffffffu, Z_l, n);
    const float aN = __shfl_sync(0xffffffffu, a_l, n);
    const float uG = __shfl_sync(0xffffffffu, ux, G);
    const float* smn = sh.slot_m + n * nchm;
    const double S = row_mass(smn, nchm, lane);
    const T* lrow = static_cast<const T*>(P.logits) + (static_cast<int64_t>(b) * R + n) * V;
    const float* qrow = (n < G) ? P.q + (static_cast<int64_t>(b) * G + n) * V : nullptr;
    int y;
    bool zr = false;
    if (!(S > 0.0)) {  // the residual of row n summed to 0 (rounding): draw from p_n
      y = draw_from_masses<T, CH>(V, nchm, nullptr, lrow, nullptr, mN, c, aN, 1.f / zN, uG, lane, zr);
      zr = true;
    } else {
      const double target = static_cast<double>(uG) * S;
      int cstar;
      double before;
      find_chunk(smn, nchm, target, lane, cstar, before);
      y = scan_chunk<T, CH>(V, lrow, qrow, mN, c, aN, qrow == nullptr, cstar, before, target, lane);
    }
    if (lane < R) tok_out[lane] = lane < n ? x : (lane == n ? y : -1);
    if (lane < G && pd_out) pd_out[lane] = px_l;
    if (lane == 0) {
      P.out_J[b] = n;
      if (P.out_status) P.out_status[b] = status | (zr ? SPECDEC_STATUS_ZERO_RESIDUAL : 0);
    }
  }

  // copies still in flight (only after a bounded wait gave up): wait for them, bounded
  for (; landed < issued; ++landed) mbar_wait(&bar[landed % kStages], (landed / kStages) & 1u);
}

template <typename T>
cudaError_t launch_row_t(const ChainParams& P, cudaStream_t stream) {
  constexpr int smem = kW * kStages * kStage;
  static unsigned long long configured = 0;
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured & bit)) {
    if (cudaError_t e = cudaFuncSetAttribute(block_row_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        e != cudaSuccess)
      return e;
    configured |= bit;
  }
  const int grid = min(device_sm_count(), P.B);
  return launch_kernel(block_row_kernel<T>, dim3(grid), dim3(kW * 32), smem, stream, 0, P);
}

}  // namespace

cudaError_t launch_block_fused(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream) {
  return ldt == SPECDEC_BF16 ? launch_row_t<uint16_t>(P, stream) : launch_row_t<float>(P, stream);
}

bool block_fused_fits(int g, int V, specdec_dtype ldt) {
  const int R = g + 1;
  if (R > kStreamMaxRows) return false;
  const int64_t row_bytes = static_cast<int64_t>(V) * (ldt == SPECDEC_BF16 ? 2 : 4);
  const int64_t nch = (row_bytes + kStatsChunkBytes - 1) / kStatsChunkBytes;
  const int cm = block_mass_chunk(ldt);
  const int64_t nchm = (V + cm - 1) / cm;
  return nch <= kBlockSlotsS && R * nchm <= kBlockSlotsM;
}

}  // namespace specdec
