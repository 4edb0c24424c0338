// Sampled token-tree verification by recursive rejection (one CTA per sequence).
//
// SD 20.5, box "Recursive rejection at a node with several children" (multi-step
// speculative sampling, Miao et al., SpecInfer): the children s_1..s_k of the current node
// were drafted independently from q.  With R_1 = p, child s_i is accepted when
// u * q(s_i) < R_i(s_i) and the walk moves to it; otherwise R_{i+1} = (R_i - q)+ normalised
// and the next child is tried; when every child is rejected (or the node is a leaf) the
// extra token is drawn from the last R by inverse CDF and the walk ends.
//
// Every residual is (p - a q)+ / S for a scalar a: R_1 = p (a = 0, S = 1), and
// (R_i - q)+ = (p - a q)+ / S - q)+ = (p - (a + S) q)+ / S, so a_{i+1} = a_i + S_i and
// S_{i+1} = sum (p - a_{i+1} q)+.  A rejection therefore costs one pass over the node's
// logits and q rows (S_{i+1}); a test needs only p(s_i) and q(s_i).  Per visited node:
//   pass 1   maximum, its lowest index, NaN detection (the greedy walk stops here)
//   pass 2   Z = sum 2^((l - m) c)
//   tests    in child order; each rejection: one residual pass (also checks the q row
//            the first time it is read whole)
//   draw     tiles in index order until the running weight passes u[0] * S
// Only the rows the walk visits are read.  When a node's logits and q rows fit in shared
// memory (V = 32000 bf16: 64 KB + 128 KB), they are staged there by bulk copies as the walk
// reaches the node, and every pass reads shared memory instead of making a round trip to
// L2 or HBM.

#include <climits>

#include "specdec_device.cuh"
#include "specdec_internal.h"

namespace specdec {

namespace {


template <typename T, int VEC, int NT, bool STAGED>
__global__ void __launch_bounds__(NT) tree_rr_kernel(const TreeParams P) {
  extern __shared__ __align__(128) unsigned char stage[];
  __shared__ float sh_f[32];
  __shared__ int sh_i[32];
  __shared__ double sh_d[32];
  __shared__ int s_y;
  __shared__ __align__(8) uint64_t sbar;
  using A = RowAccess<T, VEC, STAGED>;
  const int64_t lbytes = (static_cast<int64_t>(P.V) * static_cast<int64_t>(sizeof(T)) + 15) / 16 * 16;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int N = P.N, V = P.V, D = P.D;
  const float Tb = __ldg(P.temps + b);
  const bool greedy = !(Tb >= SPECDEC_GREEDY_TEMPERATURE);
  const float c = greedy ? 0.f : kLog2e / Tb;
  const int32_t* toks = P.node_tokens + static_cast<int64_t>(b) * N;
  const float* ub = P.u + static_cast<int64_t>(b) * (N + 1);
  int32_t* out_t = P.out_tokens + static_cast<int64_t>(b) * (D + 1);
  int32_t* out_p = P.out_path + static_cast<int64_t>(b) * D;
  auto row_off = [&](int node) { return (static_cast<int64_t>(b) * (N + 1) + (node < 0 ? 0 : 1 + node)) * V; };
  auto issue_rows = [&](int node, bool with_q) {  // one thread: the node's rows into the stage
    fence_proxy_async_smem();
    const int64_t roff = row_off(node);
    const char* lsrc = reinterpret_cast<const char*>(static_cast<const T*>(P.logits) + roff);
    const char* qsrc = reinterpret_cast<const char*>(P.q + roff);
    const uint32_t lb = static_cast<uint32_t>(static_cast<int64_t>(V) * sizeof(T));
    const uint32_t qb = with_q ? static_cast<uint32_t>(V) * 4u : 0u;
    mbar_expect_tx(&sbar, lb + qb);
    for (uint32_t o = 0; o < lb; o += kStageCopy)
      bulk_copy_g2s(stage + o, lsrc + o, min(static_cast<uint32_t>(kStageCopy), lb - o), &sbar);
    for (uint32_t o = 0; o < qb; o += kStageCopy)
      bulk_copy_g2s(stage + lbytes + o, qsrc + o, min(static_cast<uint32_t>(kStageCopy), qb - o), &sbar);
  };
  if constexpr (STAGED) {
    // The root's rows are read by every walk that passes validation; in a valid tree node 0
    // is a child of the root, so its q row is needed whenever N > 0 and the walk samples.
    if (tid == 0) {
      mbar_init(&sbar, 1);
      mbar_fence_init();
      issue_rows(-1, N > 0 && !greedy);
    }
  }

  // Validate the tree, the tokens, the temperature and (sampled) every uniform.
  int st = 0;
  for (int j = tid; j < N; j += NT) {
    const int a = __ldg(P.parents + j);
    if (!(a >= -1 && a < j)) st |= SPECDEC_STATUS_BAD_TREE;
    const int t = __ldg(toks + j);
    if (t < 0 || t >= V) st |= SPECDEC_STATUS_BAD_TOKEN;
  }
  st = Block<NT>::or_int(st, sh_i);
  if (!(st & SPECDEC_STATUS_BAD_TREE)) {
    int deep = 0;
    for (int j = tid; j < N; j += NT) {  // nodes on the root path of j (bounded walk)
      int a = j, cnt = 0;
      while (a >= 0 && cnt <= D) { ++cnt; a = __ldg(P.parents + a); }
      if (cnt > D) deep = SPECDEC_STATUS_BAD_TREE;
    }
    st |= Block<NT>::or_int(deep, sh_i);
  }
  if (tid == 0 && !(Tb - Tb == 0.f)) st |= SPECDEC_STATUS_BAD_TEMPERATURE;
  if (!greedy) {
    int bu = 0;
    for (int j = tid; j <= N; j += NT) {
      const float uu = __ldg(ub + j);
      if (!(uu >= 0.f && uu < 1.f)) bu = SPECDEC_STATUS_BAD_UNIFORM;
    }
    st |= bu;
  }
  st = Block<NT>::or_int(st, sh_i);

  uint32_t sphase = 0;
  if constexpr (STAGED) {  // the root copies land before the CTA reads the stage or exits
    if (Block<NT>::or_int(mbar_wait(&sbar, sphase) ? 0 : 1, sh_i)) st |= SPECDEC_STATUS_TIMEOUT;
    sphase ^= 1u;
  }
  int node = -1, d = 0;
  if (!(st & SPECDEC_STATUS_ERROR_MASK)) {
    for (;;) {
      const int64_t roff = row_off(node);
      const T* lrow = static_cast<const T*>(P.logits) + roff;
      const float* qrow = P.q + roff;
      if constexpr (STAGED) {  // bring the node's rows into shared memory (q only if it has children)
        if (node >= 0) {
          int kids = 0;
          for (int j = tid; j < N; j += NT) kids |= (__ldg(P.parents + j) == node) ? 1 : 0;
          kids = Block<NT>::or_int(kids, sh_i);  // also orders every earlier read of the stage
          if (tid == 0) issue_rows(node, kids && !greedy);
          if (Block<NT>::or_int(mbar_wait(&sbar, sphase) ? 0 : 1, sh_i)) {  // uniform decision
            st |= SPECDEC_STATUS_TIMEOUT;
            break;
          }
          sphase ^= 1u;
        }
        lrow = reinterpret_cast<const T*>(stage);
        qrow = reinterpret_cast<const float*>(stage + lbytes);
      }
      // pass 1: maximum and its lowest index (each thread walks its vectors in index order)
      float best = -kInf;
      int bidx = INT_MAX;
      bool nan = false;
      for (int k = tid * VEC; k < V; k += NT * VEC) {
        float v[VEC];
        A::vec(lrow, k, v);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          nan |= (v[e] != v[e]);
          if (v[e] > best) { best = v[e]; bidx = k + e; }  // strict: first index kept on ties
        }
      }
      if (nan) best = __int_as_float(0x7fc00000);
      const float m = Block<NT>::max(best, sh_f);
      const int z = Block<NT>::min_int((best == m) ? bidx : INT_MAX, sh_i);
      int rs = 0;
      if (!(m == m) || m == kInf) rs = SPECDEC_STATUS_BAD_LOGIT;
      else if (m == -kInf) rs = SPECDEC_STATUS_EMPTY_ROW;
      if (rs) { st |= rs; break; }

      int child = INT_MAX, y = z;
      if (greedy) {  // the lowest-index child carrying the argmax
        for (int j = tid; j < N; j += NT)
          if (__ldg(P.parents + j) == node && __ldg(toks + j) == z) child = min(child, j);
        child = Block<NT>::min_int(child, sh_i);
      } else {
        // pass 2: Z (fp32 within a thread and a warp, fp64 across warps)
        float zt = 0.f;
        for (int k = tid * VEC; k < V; k += NT * VEC) {
          float v[VEC];
          A::vec(lrow, k, v);
          float a = 0.f;
#pragma unroll
          for (int e = 0; e < VEC; ++e) a += ex2((v[e] - m) * c);
          zt += a;
        }
        const double Zd = Block<NT>::sum_f(zt, sh_d);
        const float invZ = static_cast<float>(1.0 / Zd);
        // the current residual is (p - a q)+ / S
        double a = 0.0, S = 1.0;
        bool q_checked = false;
        int prev = -1;
        for (;;) {
          int j = INT_MAX;  // the next child in index order
          for (int i = prev + 1 + tid; i < N; i += NT)
            if (__ldg(P.parents + i) == node) { j = i; break; }
          j = Block<NT>::min_int(j, sh_i);
          if (j == INT_MAX) break;
          prev = j;
          const int s = __ldg(toks + j);
          const float qs = A::qone(qrow, s);
          if (!(qs >= 0.f && qs < kInf)) { st |= SPECDEC_STATUS_BAD_PROB; break; }
          const float ps = ex2((A::one(lrow, s) - m) * c) * invZ;
          const double Rs = fmax(static_cast<double>(ps) - a * static_cast<double>(qs), 0.0) / S;
          bool accept;
          if (qs == 0.f) {
            st |= SPECDEC_STATUS_ZERO_Q;
            accept = Rs > 0.0;
          } else {
            accept = static_cast<double>(__ldg(ub + 1 + j)) * static_cast<double>(qs) < Rs;
          }
          if (accept) { child = j; break; }
          // rejected: S' = sum (p - (a + S) q)+, and the q row is read whole
          const double an = a + S;
          const float anf = static_cast<float>(an);
          float rt = 0.f;
          int qbad = 0;
          for (int k = tid * VEC; k < V; k += NT * VEC) {
            float v[VEC], qv[VEC];
            A::vec(lrow, k, v);
            A::qvec(qrow, k, qv);
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
              if (!(qv[e] >= 0.f && qv[e] < kInf)) qbad = 1;
              acc += fmaxf(ex2((v[e] - m) * c) * invZ - anf * qv[e], 0.f);
            }
            rt += acc;
          }
          if (!q_checked) {
            qbad = Block<NT>::or_int(qbad, sh_i);
            if (qbad) { st |= SPECDEC_STATUS_BAD_PROB; break; }
            q_checked = true;
          }
          const double Sn = Block<NT>::sum_f(rt, sh_d);
          if (Sn > 0.0) {
            a = an;
            S = Sn;
          } else {
            st |= SPECDEC_STATUS_ZERO_RESIDUAL;  // keep R_i (rounding only)
          }
        }
        if (st & SPECDEC_STATUS_ERROR_MASK) break;
        if (child == INT_MAX) {
          // the draw: weights 2^((l - m)c) (a = 0: p unnormalised, total from pass 2) or
          // (p - a q)+ (total S); tiles of NT vectors until the running weight passes u[0] * S
          const bool resid = a > 0.0;
          const float af = static_cast<float>(a);
          const double total = resid ? S : Zd;
          const double target = static_cast<double>(__ldg(ub)) * total;
          double base = 0.0;
          if (tid == 0) s_y = -1;
          int last_pos = -1;
          for (int k0 = 0; k0 < V; k0 += NT * VEC) {
            const int k = k0 + tid * VEC;
            float w[VEC];
            float acc = 0.f;
            if (k < V) {
              float v[VEC], qv[VEC];
              A::vec(lrow, k, v);
              if (resid) A::qvec(qrow, k, qv);
#pragma unroll
              for (int e = 0; e < VEC; ++e) {
                const float ex = ex2((v[e] - m) * c);
                w[e] = resid ? fmaxf(ex * invZ - af * qv[e], 0.f) : ex;
                acc += w[e];
                if (w[e] > 0.f) last_pos = k + e;
              }
            } else {
#pragma unroll
              for (int e = 0; e < VEC; ++e) w[e] = 0.f;
            }
            double tile;
            const double incl = Block<NT>::inclusive_scan_f(acc, sh_d, tile);
            if (base + tile > target) {
              const int first = Block<NT>::min_int((base + incl > target) ? tid : INT_MAX, sh_i);
              if (tid == first) {
                const double excl = base + (incl - static_cast<double>(acc));
                float run = 0.f;
                int yy = -1, lp = -1;
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                  run += w[e];
                  if (w[e] > 0.f) lp = k + e;
                  if (yy < 0 && excl + static_cast<double>(run) > target) yy = k + e;
                }
                s_y = (yy >= 0) ? yy : lp;
              }
              __syncthreads();
              break;
            }
            base += tile;
          }
          __syncthreads();
          y = s_y;
          if (y < 0) y = -Block<NT>::min_int(last_pos < 0 ? INT_MAX : -last_pos, sh_i);
        }
      }
      if (child == INT_MAX) {
        if (tid == 0) out_t[d] = y;
        break;
      }
      if (tid == 0) {
        out_t[d] = __ldg(toks + child);
        out_p[d] = child;
      }
      node = child;
      ++d;
    }
  }

  const bool err = (st & SPECDEC_STATUS_ERROR_MASK) != 0;
  for (int i = tid; i <= D; i += NT)
    if (err || i > d) out_t[i] = -1;
  for (int i = tid; i < D; i += NT)
    if (err || i >= d) out_p[i] = -1;
  if (tid == 0) {
    P.out_J[b] = err ? -1 : d;
    if (P.out_status) P.out_status[b] = err ? (st & SPECDEC_STATUS_ERROR_MASK) : st;
  }
}

template <typename T, int VEC, bool STAGED>
cudaError_t launch_rr_t(const TreeParams& P, cudaStream_t stream) {
  int smem = 0;
  if constexpr (STAGED) {
    smem = static_cast<int>((static_cast<int64_t>(P.V) * static_cast<int64_t>(sizeof(T)) + 15) / 16 * 16 +
                            static_cast<int64_t>(P.V) * 4);
    static unsigned long long configured = 0;
    int dev = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(configured & bit)) {
      if (cudaError_t e = cudaFuncSetAttribute(tree_rr_kernel<T, VEC, kTreeThreads, true>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, kTreeStageBytes);
          e != cudaSuccess)
        return e;
      configured |= bit;
    }
  }
  return launch_kernel(tree_rr_kernel<T, VEC, kTreeThreads, STAGED>, dim3(P.B), dim3(kTreeThreads),
                       static_cast<size_t>(smem), stream, 0, P);
}

}  // namespace

cudaError_t launch_tree_rr(const TreeParams& P, specdec_dtype ldt, bool vector_path, cudaStream_t stream) {
  if (vector_path) {
    const int64_t need = (static_cast<int64_t>(P.V) * (ldt == SPECDEC_BF16 ? 2 : 4) + 15) / 16 * 16 +
                         static_cast<int64_t>(P.V) * 4;
    if (need <= kTreeStageBytes) {
      if (ldt == SPECDEC_BF16) return launch_rr_t<uint16_t, 8, true>(P, stream);
      return launch_rr_t<float, 4, true>(P, stream);
    }
    if (ldt == SPECDEC_BF16) return launch_rr_t<uint16_t, 8, false>(P, stream);
    return launch_rr_t<float, 4, false>(P, stream);
  }
  if (ldt == SPECDEC_BF16) return launch_rr_t<uint16_t, 1, false>(P, stream);
  return launch_rr_t<float, 1, false>(P, stream);
}

}  // namespace specdec
