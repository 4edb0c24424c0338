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
//   row      maximum, its lowest index and NaN detection (the greedy walk stops here),
//            then Z = sum 2^((l - m) c) relative to each thread's maximum, combined over
//            warps by rescaling; warp 0 lists the node's children in index order
//   tests    in child order, taken alike by every thread; each rejection: one residual
//            pass (which also checks the q row the first time it is read whole)
//   draw     the warp whose chunk holds u[0] * S (from the per-warp masses of the last
//            pass) scans that chunk in index order
// Each warp owns a contiguous chunk of the row, read by its lanes as consecutive vectors,
// so per-warp masses are prefix blocks of the row.  Masses are fp32 (fp64 is slow on this
// part and this path is a chain of dependent steps): a prefix carries at most a few dozen
// roundings, a few 1e-6 relative, below the 1e-5 band in which the parity rule treats a
// boundary as a tie; totals and prefixes are summed in the same warp order, so they agree.
// Children drawn without replacement (P.wor; Sequoia): try i tests against q_i, q with the
// rejected siblings' tokens zeroed and renormalised by Z_i = 1 - (q at them).  The residual
// form stays (p - a q)+ / S with the raw q: (R_i - q_i)+ = (p - (a + S / Z_i) q)+ / S at
// every token not yet rejected, and a rejected token already has p - a q < 0 (it was
// rejected because R_i(s) < q_i(s)), so a_{i+1} = a_i + S_i / Z_i.  Z_i is kept in fp64 (a
// few subtractions per node).  When Z_i <= 0, q_i is zero: the ZERO_Q test, no pass.
// Only the rows the walk visits are read.  When a node's logits and q rows fit in shared
// memory (V = 32000 bf16: 64 KB + 128 KB), they are staged there by bulk copies as the walk
// reaches the node, and every pass reads shared memory instead of making a round trip to
// L2 or HBM.

#include <climits>

#include "specdec_device.cuh"
#include "specdec_internal.h"

namespace specdec {

namespace {

constexpr int kRRKids = 256;  // children of one node listed in shared memory at a time

template <typename T, int VEC, int NT, bool STAGED>
__global__ void __launch_bounds__(NT, 2) tree_rr_kernel(const TreeParams P) {
  constexpr int WARPS = NT / 32;
  constexpr int SPAN = 32 * VEC;  // elements per warp iteration
  constexpr unsigned FULL = 0xffffffffu;
  static_assert(WARPS <= 32, "one lane per warp in the cross-warp steps");
  extern __shared__ __align__(128) unsigned char stage[];
  __shared__ int sh_i[32];
  __shared__ int s_vp[NT], s_vt[NT];  // validation without replacement: (parent, token) per node
  __shared__ unsigned long long s_key[32];
  __shared__ float s_wz[32];     // per-warp mass of the current pass
  __shared__ float s_dw[32];     // per-warp mass of the weights the draw uses
  __shared__ int s_qbad[2][32];
  __shared__ float s_wr[2][32];  // per-warp residual mass of a rejection's pass, by parity
  __shared__ int s_kids[kRRKids];
  __shared__ int s_nkids, s_more, s_y, s_ow;
  __shared__ float s_m, s_Z, s_dbase;
  __shared__ int s_z, s_rs;
  __shared__ __align__(8) uint64_t sbar;
  using A = RowAccess<T, VEC, STAGED>;
  const int64_t lbytes = (static_cast<int64_t>(P.V) * static_cast<int64_t>(sizeof(T)) + 15) / 16 * 16;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = P.N, V = P.V, D = P.D;
  const int wchunk = ((V + WARPS - 1) / WARPS + SPAN - 1) / SPAN * SPAN;
  const int w0 = min(V, warp * wchunk), w1 = min(V, warp * wchunk + wchunk);
  const float Tb = __ldg(P.temps + b);
  const bool greedy = !(Tb >= SPECDEC_GREEDY_TEMPERATURE);
  const float c = greedy ? 0.f : kLog2e / Tb;
  const int32_t* toks = P.node_tokens + static_cast<int64_t>(b) * N;
  const float* ub = P.u + static_cast<int64_t>(b) * (N + 1);
  int32_t* out_t = P.out_tokens + static_cast<int64_t>(b) * (D + 1);
  int32_t* out_p = P.out_path + static_cast<int64_t>(b) * D;
  auto row_off = [=](int node) { return (static_cast<int64_t>(b) * (N + 1) + (node < 0 ? 0 : 1 + node)) * V; };
  auto issue_rows = [=](int node, bool with_q) {  // one thread: the node's rows into the stage
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
  // Warp 0: the children of `node` with index above `after`, in index order, into s_kids
  // (s_more: more remain beyond the list).
  auto list_kids = [=](int node, int after) {
    int n = 0;
    bool full = false;  // the list filled up: children may remain after its last entry
    for (int j0 = after + 1; j0 < N; j0 += 32) {
      const int j = j0 + lane;
      const bool is = j < N && __ldg(P.parents + j) == node;
      const unsigned bal = __ballot_sync(FULL, is);
      const int pos = n + __popc(bal & ((1u << lane) - 1u));
      if (is && pos < kRRKids) s_kids[pos] = j;
      n += __popc(bal);
      if (n >= kRRKids) {
        full = true;
        break;
      }
    }
    if (lane == 0) {
      s_nkids = min(n, kRRKids);
      s_more = full ? 1 : 0;
    }
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
    if (P.wor && N <= NT) {  // (parent, token) pairs for the repeated-sibling check below
      s_vp[j] = a;
      s_vt[j] = t;
    } else if (P.wor) {
      st |= sibling_repeats(P.parents, toks, j, a, t);
    }
  }
  if (P.wor && N <= NT) {
    __syncthreads();
    if (tid < N) st |= sibling_repeats_staged(s_vp, s_vt, tid);
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
      // ---- the row: maximum and its lowest index, and (sampled) Z relative to each
      // thread's maximum; warps combine by rescaling to the warp maximum ----------------
      float best = -kInf, zs = 0.f;
      int bidx = INT_MAX;
      bool nan = false;
      for (int k = w0 + lane * VEC; k < w1; k += SPAN) {  // each thread visits its indices in order
        float v[VEC];
        A::vec(lrow, k, v);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          nan |= (v[e] != v[e]);
          if (v[e] > best) { best = v[e]; bidx = k + e; }
        }
      }
      if (!greedy && best > -kInf && !nan)
        for (int k = w0 + lane * VEC; k < w1; k += SPAN) {
          float v[VEC];
          A::vec(lrow, k, v);
#pragma unroll
          for (int e = 0; e < VEC; ++e)
            if (v[e] > -kInf) zs += ex2((v[e] - best) * c);
        }
      const unsigned long long wk = warp_max_key(order_key(best, bidx, nan));
      if (!greedy) {
        const float wm = key_value(wk);
        float zw = best > -kInf ? zs * ex2((best - wm) * c) : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) zw += __shfl_xor_sync(FULL, zw, o);
        if (lane == 0) s_wz[warp] = zw;
      }
      if (lane == 0) s_key[warp] = wk;
      __syncthreads();
      if (warp == 0) {  // the row's maximum, Z in warp order, and this node's children
        const unsigned long long kl = lane < WARPS ? s_key[lane] : 0ull;
        const unsigned long long K = warp_max_key(kl);
        const float m = key_value(K);
        int rs = 0;
        if (!(m == m) || m == kInf) rs = SPECDEC_STATUS_BAD_LOGIT;
        else if (m == -kInf) rs = SPECDEC_STATUS_EMPTY_ROW;
        if (!greedy && rs == 0 && lane < WARPS) {  // per-warp weights 2^((l - m) c), the a = 0 draw's
          const float kv = key_value(kl);
          s_dw[lane] = kv > -kInf ? s_wz[lane] * ex2((kv - m) * c) : 0.f;
        }
        __syncwarp();
        list_kids(node, -1);
        if (lane == 0) {
          float Z = 0.f;
          if (!greedy && rs == 0)
            for (int w = 0; w < WARPS; ++w) Z += s_dw[w];
          s_rs = rs;
          s_m = m;
          s_z = key_index(K);
          s_Z = Z;
        }
      }
      __syncthreads();
      if (s_rs) {
        st |= s_rs;
        break;
      }
      const float m = s_m;

      int child = INT_MAX, y = s_z;
      if (greedy) {  // the lowest-index child carrying the argmax
        if (!s_more) {
          for (int i = 0; i < s_nkids; ++i)
            if (__ldg(toks + s_kids[i]) == y) { child = s_kids[i]; break; }
        } else {
          for (int j = tid; j < N; j += NT)
            if (__ldg(P.parents + j) == node && __ldg(toks + j) == y) child = min(child, j);
          child = Block<NT>::min_int(child, sh_i);
        }
      } else {
        const float Z = s_Z, invZ = 1.f / Z;
        // the current residual is (p - a q)+ / S
        float a = 0.f, S = 1.f;
        MassLeft zq;  // without replacement: q's mass left at this node
        bool q_checked = false;
        int ki = 0, par = 0;
        for (;;) {
          if (ki == s_nkids) {  // the listed children are done
            if (!s_more) break;
            const int after = s_kids[s_nkids - 1];
            __syncthreads();  // every thread has read the list
            if (warp == 0) list_kids(node, after);
            __syncthreads();
            ki = 0;
            continue;
          }
          const int j = s_kids[ki++];
          const int s = __ldg(toks + j);
          const float qraw = A::qone(qrow, s);
          if (!(qraw >= 0.f && qraw < kInf)) { st |= SPECDEC_STATUS_BAD_PROB; break; }
          // this try's q(s): as given, or q_i(s) without replacement
          const float zv = zq.value();
          const float qs = !P.wor ? qraw : (zv > 0.f ? qraw / zv : 0.f);
          const float ps = ex2((A::one(lrow, s) - m) * c) * invZ;
          const float Rs = fmaxf(ps - a * qraw, 0.f) / S;
          bool accept;
          if (qs == 0.f) {
            st |= SPECDEC_STATUS_ZERO_Q;
            accept = Rs > 0.f;
          } else {
            accept = __ldg(ub + 1 + j) * qs < Rs;
          }
          if (accept) { child = j; break; }
          if (P.wor) {
            zq.sub(qraw);
            if (!(zv > 0.f)) continue;  // q_i = 0: the residual stays R_i
          }
          // rejected: S' = sum (p - (a + S / Z_i) q)+, and the q row is read whole
          const float an = a + (P.wor ? S / zv : S);
          float rt = 0.f;
          int qbad = 0;
          for (int k = w0 + lane * VEC; k < w1; k += SPAN) {
            float v[VEC], qv[VEC];
            A::vec(lrow, k, v);
            A::qvec(qrow, k, qv);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
              if (!(qv[e] >= 0.f && qv[e] < kInf)) qbad = 1;
              rt += fmaxf(ex2((v[e] - m) * c) * invZ - an * qv[e], 0.f);
            }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) rt += __shfl_xor_sync(FULL, rt, o);
          qbad = __any_sync(FULL, qbad) ? 1 : 0;
          if (lane == 0) {
            s_wr[par][warp] = rt;
            s_qbad[par][warp] = qbad;
          }
          __syncthreads();
          float Sn = 0.f;  // in warp order, so every thread holds the same bits
          int qb = 0;
          for (int w = 0; w < WARPS; ++w) {
            Sn += s_wr[par][w];
            qb |= s_qbad[par][w];
          }
          if (!q_checked) {
            if (qb) { st |= SPECDEC_STATUS_BAD_PROB; break; }
            q_checked = true;
          }
          if (Sn > 0.f) {
            a = an;
            S = Sn;
            if (tid < WARPS) s_dw[tid] = s_wr[par][tid];  // the draw's per-warp weights now
          } else {
            st |= SPECDEC_STATUS_ZERO_RESIDUAL;  // keep R_i (rounding only)
          }
          par ^= 1;
        }
        if (st & SPECDEC_STATUS_ERROR_MASK) break;
        if (child == INT_MAX) {
          // the draw: weights 2^((l - m)c) (a = 0: total Z) or (p - a q)+ (total S); the warp
          // whose chunk holds u[0] * total scans it in index order
          const bool resid = a > 0.f;
          const float total = resid ? S : Z;
          const float target = __ldg(ub) * total;
          __syncthreads();  // s_dw is complete
          if (tid == 0) {  // prefix in warp order, as the totals were summed
            float base = 0.f, lastb = 0.f;
            int ow = -1, lastw = -1;
            for (int w = 0; w < WARPS; ++w) {
              const float x = s_dw[w];
              if (x > 0.f) { lastw = w; lastb = base; }
              if (ow < 0 && base + x > target) { ow = w; s_dbase = base; }
              base += x;
            }
            if (ow < 0) {  // past the end only by rounding: the last warp with mass
              ow = lastw < 0 ? 0 : lastw;
              s_dbase = lastb;
            }
            s_ow = ow;
            s_y = -1;
          }
          __syncthreads();
          if (warp == s_ow) {
            float base = s_dbase;
            int yy = -1, wl = -1;
            for (int k0 = w0; k0 < w1; k0 += SPAN) {
              const int k = k0 + lane * VEC;
              float wt[VEC];
              float acc = 0.f;
              if (k < w1) {
                float v[VEC], qv[VEC];
                A::vec(lrow, k, v);
                if (resid) A::qvec(qrow, k, qv);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                  const float ex = ex2((v[e] - m) * c);
                  wt[e] = resid ? fmaxf(ex * invZ - a * qv[e], 0.f) : ex;
                  acc += wt[e];
                  if (wt[e] > 0.f) wl = k + e;
                }
              } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) wt[e] = 0.f;
              }
              float incl = acc;
#pragma unroll
              for (int o = 1; o < 32; o <<= 1) {
                const float t = __shfl_up_sync(FULL, incl, o);
                if (lane >= o) incl += t;
              }
              const float rem = target - base;  // mass still to pass at this tile's start
              const unsigned hit = __ballot_sync(FULL, incl > rem);
              if (hit) {
                const int first = __ffs(hit) - 1;
                if (lane == first) {
                  const float excl = incl - acc;
                  float run = 0.f;
                  int lp = -1;
#pragma unroll
                  for (int e = 0; e < VEC; ++e) {
                    run += wt[e];
                    if (wt[e] > 0.f) lp = k + e;
                    if (yy < 0 && excl + run > rem) yy = k + e;
                  }
                  if (yy < 0) yy = lp;
                }
                yy = __shfl_sync(FULL, yy, first);
                break;
              }
              base += __shfl_sync(FULL, incl, 31);
            }
            wl = __reduce_max_sync(FULL, wl);
            if (yy < 0) yy = wl;  // the chunk ended before the point by rounding
            if (lane == 0) s_y = yy;
          }
          __syncthreads();
          y = s_y;
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
