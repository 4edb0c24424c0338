// Recursive rejection at multi-child tree nodes, with each row split across a cluster.
//
// SD 20.5, box "Recursive rejection at a node with several children" (multi-step
// speculative sampling, Miao et al., SpecInfer): the children s_1..s_k of the current node
// were drafted independently from q.  With R_1 = p, child s_i is accepted when
// u * q(s_i) < R_i(s_i) and the walk moves to it; otherwise R_{i+1} = (R_i - q)+ normalised
// and the next child is tried; when every child is rejected (or the node is a leaf) the
// extra token is drawn from the last R by inverse CDF and the walk ends.  Every residual is
// (p - a q)+ / S for a scalar a (a_1 = 0, S_1 = 1; a rejection gives a <- a + S and
// S <- sum (p - a q)+), so a test needs only p(s_i) and q(s_i), and a rejection costs one
// pass over the node's logits and q rows.  Children drawn without replacement (P.wor;
// Sequoia) test against q_i = q off the rejected siblings' tokens, renormalised by
// Z_i = 1 - (q at them); the residual keeps its form with the raw q and a <- a + S / Z_i
// (a rejected token already has p - a q < 0); Z_i in fp64; Z_i <= 0: q_i = 0, no pass.
//
// A cluster of C CTAs serves one sequence (as the Medusa walk of tree_walk_cluster.cu):
// CTA r stages the contiguous slice r of the visited node's logits row (and q row, when
// the node has children) with bulk copies.  Per visited node:
//   entry    warp 0 lists the node's children in index order and loads the logit and q
//            at each child's token (every CTA alike: the tests need them everywhere)
//   row      the slice's maximum and lowest index (64-bit order key) and Z relative to
//            each thread's maximum, combined over warps                       -> mail A
//            every CTA merges the C messages in rank order: m, Z, the row status
//   tests    in child order, taken alike by every thread of every CTA; a rejection is a
//            residual pass over the slice                                      -> mail B
//   draw     the CTA, then the warp chunk, holding u[0] * S; one warp scans it  -> mail C
// Mail is one 16-byte message per CTA pushed into every member's shared memory with
// st.async (all-to-all; two parities; see tree_walk_cluster.cu for why no slot is
// rewritten early).  Masses are fp32: a prefix carries at most a few dozen roundings, a
// few 1e-6 relative, below the 1e-5 band in which the parity rule treats a boundary as a
// tie.  Waiting lanes enter their polling loop converged.  Inputs are validated up front
// (the walk starts after); the root's copies are issued before validation.

#include <climits>

#include "specdec_device.cuh"
#include "specdec_internal.h"

namespace specdec {

namespace {

constexpr int kRRCopy = 32768;    // bytes per bulk copy
constexpr int kRRMaxC = 8;
constexpr int kRRKidsC = 256;     // children of one node listed at a time
constexpr unsigned kAll = 0xffffffffu;

struct RRShared {
  uint4 slot[2][kRRMaxC];           // mailbox: one 16-byte message per member, by parity
  uint64_t xbar[2];                 // mailbox barriers, by parity
  uint64_t sbar;                    // stage barrier
  unsigned long long key[32];       // per-warp order keys of the row pass
  float wz[32];                     // per-warp Z relative to the warp maximum
  float wr[2][32];                  // per-warp residual masses of a rejection's pass, by parity
  int qbad[2][32];                  // per-warp bad-q flags of that pass, by parity
  float dw[32];                     // per-warp masses of the weights the draw uses
  float cm[kRRMaxC];                // per-CTA masses of those weights (rank order)
  int kids[kRRKidsC];               // this node's children, index order
  float kl[kRRKidsC], kq[kRRKidsC]; // the logit and q at each listed child's token
  int nkids, more;
  float m, Z, S, a;                 // row maximum, normaliser, residual total and scalar
  int z, rs, owner, ow, y, rej_bad;
  float target, obase, wbase;
};

template <typename T>
__device__ __forceinline__ void slice_vec(const T* p, int k, float (&v)[16 / sizeof(T)]) {
  if constexpr (sizeof(T) == 2) {
    const uint4 w = *reinterpret_cast<const uint4*>(p + k);
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
  } else {
    const float4 w = *reinterpret_cast<const float4*>(p + k);
    v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
  }
}
template <int N>
__device__ __forceinline__ void slice_q(const float* p, int k, float (&v)[N]) {
#pragma unroll
  for (int j = 0; j < N; j += 4) {
    const float4 w = *reinterpret_cast<const float4*>(p + k + j);
    v[j] = w.x; v[j + 1] = w.y; v[j + 2] = w.z; v[j + 3] = w.w;
  }
}

// Inclusive prefix over lanes 0..width-1 (width a power of two; a fixed tree of fp32 adds,
// so every warp running it on the same values gets the same bits).
__device__ __forceinline__ float lanes_scan(float x, int lane, int width) {
  for (int o = 1; o < width; o <<= 1) {
    const float n = __shfl_up_sync(kAll, x, o);
    if (lane >= o) x += n;
  }
  return x;
}

__device__ __forceinline__ void rr_mail(RRShared& sh, int par, uint32_t C, uint32_t rank, uint4 msg) {
  mbar_expect_tx(&sh.xbar[par], C * 16u);
  const uint32_t sa = smem_addr(&sh.slot[par][rank]);
  const uint32_t ba = smem_addr(&sh.xbar[par]);
  const float4 w = make_float4(__uint_as_float(msg.x), __uint_as_float(msg.y), __uint_as_float(msg.z),
                               __uint_as_float(msg.w));
  for (uint32_t r = 0; r < C; ++r) st_async_16(cluster_map(sa, r), w, cluster_map(ba, r));
}

template <typename T, int NT>
__global__ void __launch_bounds__(NT, 2) tree_rr_cluster_kernel(const TreeParams P, int slice, int qoff) {
  constexpr int VEC = 16 / static_cast<int>(sizeof(T));
  constexpr int WARPS = NT / 32;
  constexpr int SPAN = 32 * VEC;  // elements per warp iteration
  static_assert(WARPS <= 32 && (WARPS & (WARPS - 1)) == 0, "a power-of-two warp count, one lane per warp");
  extern __shared__ __align__(128) unsigned char stage[];
  __shared__ RRShared sh;
  __shared__ int sh_i[32];
  __shared__ int s_vp[NT], s_vt[NT];  // validation without replacement: (parent, token) per node
  const T* sl = reinterpret_cast<const T*>(stage);                 // this slice of the logits row
  const float* sq = reinterpret_cast<const float*>(stage + qoff);  // this slice of the q row
  const uint32_t C = cluster_size(), rank = cluster_rank();
  const int b = static_cast<int>(blockIdx.x / C);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = P.N, V = P.V, D = P.D;
  const int s0 = static_cast<int>(rank) * slice;
  const int n = max(0, min(V, s0 + slice) - s0);
  const int wchunk = ((n + WARPS - 1) / WARPS + SPAN - 1) / SPAN * SPAN;
  const int w0 = min(n, warp * wchunk), w1 = min(n, warp * wchunk + wchunk);
  const float Tb = __ldg(P.temps + b);
  const bool greedy = !(Tb >= SPECDEC_GREEDY_TEMPERATURE);
  const float c = greedy ? 0.f : kLog2e / Tb;
  const int32_t* toks = P.node_tokens + static_cast<int64_t>(b) * N;
  const float* ub = P.u + static_cast<int64_t>(b) * (N + 1);
  auto row_off = [=](int node) { return (static_cast<int64_t>(b) * (N + 1) + (node < 0 ? 0 : 1 + node)) * V; };
  auto issue = [=](int node, bool with_q) {  // one thread: this CTA's slices of the node's rows
    fence_proxy_async_smem();
    const int64_t roff = row_off(node) + s0;
    const char* lsrc = reinterpret_cast<const char*>(static_cast<const T*>(P.logits) + roff);
    const char* qsrc = reinterpret_cast<const char*>(P.q + roff);
    const uint32_t lb = static_cast<uint32_t>(n) * static_cast<uint32_t>(sizeof(T));
    const uint32_t qb = with_q ? static_cast<uint32_t>(n) * 4u : 0u;
    mbar_expect_tx(&sh.sbar, lb + qb);
    for (uint32_t o = 0; o < lb; o += kRRCopy)
      bulk_copy_g2s(stage + o, lsrc + o, min(static_cast<uint32_t>(kRRCopy), lb - o), &sh.sbar);
    for (uint32_t o = 0; o < qb; o += kRRCopy)
      bulk_copy_g2s(stage + qoff + o, qsrc + o, min(static_cast<uint32_t>(kRRCopy), qb - o), &sh.sbar);
  };
  // Warp 0: the children of `node` after index `after`, in index order, and (sampled) the
  // logit and q at each one's token, read from global memory (the slice of a token may
  // belong to another CTA).
  auto list_kids = [=](int node, int after) {
    int cnt = 0;
    bool full = false;
    for (int j0 = after + 1; j0 < N; j0 += 32) {
      const int j = j0 + lane;
      const bool is = j < N && __ldg(P.parents + j) == node;
      const unsigned bal = __ballot_sync(kAll, is);
      const int pos = cnt + __popc(bal & ((1u << lane) - 1u));
      if (is && pos < kRRKidsC) sh.kids[pos] = j;
      cnt += __popc(bal);
      if (cnt >= kRRKidsC) {
        full = true;
        break;
      }
    }
    cnt = min(cnt, kRRKidsC);
    __syncwarp();
    if (!greedy) {
      const int64_t roff = row_off(node);
      for (int i = lane; i < cnt; i += 32) {
        const int s = __ldg(toks + sh.kids[i]);
        sh.kl[i] = Elem<T>::load(static_cast<const T*>(P.logits) + roff, s);
        sh.kq[i] = __ldg(P.q + roff + s);
      }
    }
    if (lane == 0) {
      sh.nkids = cnt;
      sh.more = full ? 1 : 0;
    }
  };
  if (tid == 0) {
    mbar_init(&sh.sbar, 1);
    mbar_init(&sh.xbar[0], 1);
    mbar_init(&sh.xbar[1], 1);
    mbar_fence_init();
    issue(-1, N > 0 && !greedy);  // in a valid tree node 0 is a child of the root
  }
  cluster_arrive_relaxed();  // the barriers exist for the other members once all arrived
  bool pending = true;       // (thread 0) a copy into the stage has not been waited for
  uint32_t sphase = 0, xk = 0;

  // Validate the tree, the tokens, the temperature and (sampled) every uniform; every CTA
  // of the cluster reaches the same status.
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
    int x = j, cnt = 0;  // nodes on the root path of j (bounded walk)
    while (x >= 0 && x < N && cnt <= D) { ++cnt; x = __ldg(P.parents + x); }
    if (cnt > D) st |= SPECDEC_STATUS_BAD_TREE;
  }
  if (!greedy)
    for (int j = tid; j <= N; j += NT) {
      const float uu = __ldg(ub + j);
      if (!(uu >= 0.f && uu < 1.f)) st |= SPECDEC_STATUS_BAD_UNIFORM;
    }
  if (tid == 0 && !(Tb - Tb == 0.f)) st |= SPECDEC_STATUS_BAD_TEMPERATURE;
  if (P.wor && N <= NT) {
    __syncthreads();
    if (tid < N) st |= sibling_repeats_staged(s_vp, s_vt, tid);
  }
  st = Block<NT>::or_int(st, sh_i);
  cluster_wait();

  int node = -1, d = 0, y = -1;
  if (!(st & SPECDEC_STATUS_ERROR_MASK)) {
    for (;;) {
      // ---- entry: the node's children, and its rows (the root's copies are in flight)
      __syncthreads();  // every read of the previous node's list and stage is done
      if (warp == 0) {
        list_kids(node, -1);
        if (node >= 0 && lane == 0) {
          issue(node, sh.nkids > 0 && !greedy);
          pending = true;
        }
      }
      const bool landed = mbar_wait(&sh.sbar, sphase);
      if (landed) {
        sphase ^= 1u;
        pending = false;
      }
      // ---- the row: slice maximum and lowest index, Z relative to each thread's maximum
      float best = -kInf, zs = 0.f;
      int bidx = INT_MAX;
      bool nan = false;
      if (landed) {
        for (int k = w0 + lane * VEC; k < w1; k += SPAN) {
          float v[VEC];
          slice_vec<T>(sl, k, v);
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            nan |= (v[e] != v[e]);
            if (v[e] > best) { best = v[e]; bidx = s0 + k + e; }
          }
        }
        if (!greedy && best > -kInf && !nan)
          for (int k = w0 + lane * VEC; k < w1; k += SPAN) {
            float v[VEC];
            slice_vec<T>(sl, k, v);
#pragma unroll
            for (int e = 0; e < VEC; ++e)
              if (v[e] > -kInf) zs += ex2((v[e] - best) * c);
          }
      }
      const unsigned long long wk = warp_max_key(landed ? order_key(best, bidx, nan) : kKeyTimeout);
      if (!greedy) {
        const float wm = key_value(wk);
        float zw = best > -kInf ? zs * ex2((best - wm) * c) : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) zw += __shfl_xor_sync(kAll, zw, o);
        if (lane == 0) sh.wz[warp] = zw;
      }
      if (lane == 0) sh.key[warp] = wk;
      __syncthreads();
      if (warp == 0) {  // mail A: the slice's key and Z; then the row's m, Z and status
        const int par = static_cast<int>(xk & 1u);
        const unsigned long long kw = lane < WARPS ? sh.key[lane] : 0ull;
        const unsigned long long ckey = warp_max_key(kw);
        const float mr = key_value(ckey);
        const float kv = key_value(kw);
        const float wrel = (!greedy && lane < WARPS && kv > -kInf) ? sh.wz[lane] * ex2((kv - mr) * c) : 0.f;
        const float zc = __shfl_sync(kAll, lanes_scan(wrel, lane, WARPS), WARPS - 1);
        if (lane == 0)
          rr_mail(sh, par, C, rank,
                  make_uint4(static_cast<uint32_t>(ckey), static_cast<uint32_t>(ckey >> 32), __float_as_uint(zc), 0u));
        __syncwarp();
        const bool ok = !__any_sync(kAll, !mbar_wait_cluster(&sh.xbar[par], (xk >> 1) & 1u));
        unsigned long long kr = 0ull;
        float zr = 0.f;
        if (lane < static_cast<int>(C)) {
          const uint4 s = sh.slot[par][lane];
          kr = (static_cast<unsigned long long>(s.y) << 32) | s.x;
          zr = __uint_as_float(s.z);
        }
        const unsigned long long K = warp_max_key(kr);
        const float m = key_value(K);
        int rs = 0;
        if (!ok || K == kKeyTimeout) rs = SPECDEC_STATUS_TIMEOUT;
        else if (!(m == m) || m == kInf) rs = SPECDEC_STATUS_BAD_LOGIT;
        else if (m == -kInf) rs = SPECDEC_STATUS_EMPTY_ROW;
        float Z = 0.f;
        if (rs == 0 && !greedy) {  // slice masses rescaled to m: Z, and the a = 0 draw's masses
          const float mk = key_value(kr);
          const float cz = (lane < static_cast<int>(C) && mk > -kInf) ? zr * ex2((mk - m) * c) : 0.f;
          Z = __shfl_sync(kAll, lanes_scan(cz, lane, static_cast<int>(C)), static_cast<int>(C) - 1);
          if (lane < static_cast<int>(C)) sh.cm[lane] = cz;
          if (lane < WARPS) sh.dw[lane] = kv > -kInf ? sh.wz[lane] * ex2((kv - m) * c) : 0.f;
        }
        if (lane == 0) {
          sh.rs = rs;
          sh.m = m;
          sh.Z = Z;
          sh.z = key_index(K);
        }
      }
      ++xk;
      __syncthreads();
      if (sh.rs) {
        st |= sh.rs;
        break;
      }
      const float m = sh.m;

      int child = INT_MAX;
      y = sh.z;
      if (greedy) {  // the lowest-index child carrying the argmax
        if (!sh.more) {
          for (int i = 0; i < sh.nkids; ++i)
            if (__ldg(toks + sh.kids[i]) == y) { child = sh.kids[i]; break; }
        } else {
          for (int j = tid; j < N; j += NT)
            if (__ldg(P.parents + j) == node && __ldg(toks + j) == y) child = min(child, j);
          child = Block<NT>::min_int(child, sh_i);
        }
      } else {
        const float Z = sh.Z, invZ = 1.f / Z;
        float a = 0.f, S = 1.f;  // the current residual is (p - a q)+ / S
        MassLeft zq;             // without replacement: q's mass left at this node
        bool q_checked = false;
        int ki = 0, par = 0;
        for (;;) {
          if (ki == sh.nkids) {  // the listed children are done
            if (!sh.more) break;
            const int after = sh.kids[sh.nkids - 1];
            __syncthreads();  // every thread has read the list
            if (warp == 0) list_kids(node, after);
            __syncthreads();
            ki = 0;
            continue;
          }
          const int j = sh.kids[ki];
          const float lj = sh.kl[ki], qraw = sh.kq[ki];
          ++ki;
          if (!(qraw >= 0.f && qraw < kInf)) { st |= SPECDEC_STATUS_BAD_PROB; break; }
          // this try's q(s): as given, or q_i(s) without replacement
          const float zv = zq.value();
          const float qs = !P.wor ? qraw : (zv > 0.f ? qraw / zv : 0.f);
          const float ps = ex2((lj - m) * c) * invZ;
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
          // rejected: the slice's part of S' = sum (p - (a + S / Z_i) q)+ (and the q check)
          const float an = a + (P.wor ? S / zv : S);
          float rt = 0.f;
          int qbad = 0;
          for (int k = w0 + lane * VEC; k < w1; k += SPAN) {
            float v[VEC], qv[VEC];
            slice_vec<T>(sl, k, v);
            slice_q<VEC>(sq, k, qv);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
              if (!(qv[e] >= 0.f && qv[e] < kInf)) qbad = 1;
              rt += fmaxf(ex2((v[e] - m) * c) * invZ - an * qv[e], 0.f);
            }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) rt += __shfl_xor_sync(kAll, rt, o);
          qbad = __any_sync(kAll, qbad) ? 1 : 0;
          if (lane == 0) {
            sh.wr[par][warp] = rt;
            sh.qbad[par][warp] = qbad;
          }
          __syncthreads();
          if (warp == 0) {  // mail B: the slice's residual mass; then S' over the cluster
            const int xp = static_cast<int>(xk & 1u);
            const float wv = lane < WARPS ? sh.wr[par][lane] : 0.f;
            const float mc = __shfl_sync(kAll, lanes_scan(wv, lane, WARPS), WARPS - 1);
            const int qc = __any_sync(kAll, lane < WARPS && sh.qbad[par][lane] != 0) ? 1 : 0;
            if (lane == 0) rr_mail(sh, xp, C, rank, make_uint4(__float_as_uint(mc), static_cast<uint32_t>(qc), 0u, 0u));
            __syncwarp();
            const bool ok = !__any_sync(kAll, !mbar_wait_cluster(&sh.xbar[xp], (xk >> 1) & 1u));
            float cr = 0.f;
            int qr = 0;
            if (lane < static_cast<int>(C)) {
              const uint4 s = sh.slot[xp][lane];
              cr = __uint_as_float(s.x);
              qr = static_cast<int>(s.y);
            }
            const float Sn = __shfl_sync(kAll, lanes_scan(cr, lane, static_cast<int>(C)), static_cast<int>(C) - 1);
            const int qall = __any_sync(kAll, qr != 0) ? 1 : 0;
            if (ok && Sn > 0.f) {  // the draw's masses are this pass's, unless a later one replaces them
              if (lane < static_cast<int>(C)) sh.cm[lane] = cr;
              if (lane < WARPS) sh.dw[lane] = wv;
            }
            if (lane == 0) {
              sh.S = Sn;
              sh.rej_bad = ok ? qall : -1;
            }
          }
          ++xk;
          __syncthreads();
          const float Sn = sh.S;
          const int rb = sh.rej_bad;
          if (rb < 0) { st |= SPECDEC_STATUS_TIMEOUT; break; }
          if (!q_checked) {
            if (rb) { st |= SPECDEC_STATUS_BAD_PROB; break; }
            q_checked = true;
          }
          if (Sn > 0.f) {
            a = an;
            S = Sn;
          } else {
            st |= SPECDEC_STATUS_ZERO_RESIDUAL;  // keep R_i (rounding only)
          }
          par ^= 1;
        }
        if (st & SPECDEC_STATUS_ERROR_MASK) break;
        if (child == INT_MAX) {
          // ---- the draw: weights 2^((l - m) c) (a = 0, total Z) or (p - a q)+ (total S)
          const bool resid = a > 0.f;
          const float target = __ldg(ub) * (resid ? S : Z);
          if (warp == 0) {  // the CTA, then (in the owner) the warp chunk, holding the point
            const float cx = lane < static_cast<int>(C) ? sh.cm[lane] : 0.f;
            const float ci = lanes_scan(cx, lane, static_cast<int>(C));
            const unsigned ch = __ballot_sync(kAll, lane < static_cast<int>(C) && ci > target);
            const unsigned cp = __ballot_sync(kAll, lane < static_cast<int>(C) && cx > 0.f);
            const int owner = ch ? __ffs(ch) - 1 : (cp ? 31 - __clz(cp) : 0);  // past the end: rounding
            const float cb = __shfl_sync(kAll, ci, owner > 0 ? owner - 1 : 0);
            const float obase = owner > 0 ? cb : 0.f;
            int ow = 0;
            float wbase = obase;
            if (owner == static_cast<int>(rank)) {
              const float wx = lane < WARPS ? sh.dw[lane] : 0.f;
              const float wi = obase + lanes_scan(wx, lane, WARPS);
              const unsigned wh = __ballot_sync(kAll, lane < WARPS && wi > target);
              const unsigned wp = __ballot_sync(kAll, lane < WARPS && wx > 0.f);
              ow = wh ? __ffs(wh) - 1 : (wp ? 31 - __clz(wp) : 0);
              const float wb = __shfl_sync(kAll, wi, ow > 0 ? ow - 1 : 0);
              wbase = ow > 0 ? wb : obase;
            }
            if (lane == 0) {
              sh.owner = owner;
              sh.ow = ow;
              sh.wbase = wbase;
            }
          }
          __syncthreads();
          const int owner = sh.owner;
          const int par = static_cast<int>(xk & 1u);
          if (owner == static_cast<int>(rank) && warp == sh.ow) {  // mail C from the owner warp
            float base = sh.wbase;
            int yy = -1, wl = -1;
            for (int k0 = w0; k0 < w1; k0 += SPAN) {
              const int k = k0 + lane * VEC;
              float wt[VEC];
              float acc = 0.f;
              if (k < w1) {
                float v[VEC], qv[VEC];
                slice_vec<T>(sl, k, v);
                if (resid) slice_q<VEC>(sq, k, qv);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                  const float ex = ex2((v[e] - m) * c);
                  wt[e] = resid ? fmaxf(ex * invZ - a * qv[e], 0.f) : ex;
                  acc += wt[e];
                  if (wt[e] > 0.f) wl = s0 + k + e;
                }
              } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) wt[e] = 0.f;
              }
              float incl = acc;
#pragma unroll
              for (int o = 1; o < 32; o <<= 1) {
                const float t = __shfl_up_sync(kAll, incl, o);
                if (lane >= o) incl += t;
              }
              const float rem = target - base;  // mass still to pass at this tile's start
              const unsigned hit = __ballot_sync(kAll, incl > rem);
              if (hit) {
                const int first = __ffs(hit) - 1;
                if (lane == first) {
                  const float excl = incl - acc;
                  float run = 0.f;
                  int lp = -1;
#pragma unroll
                  for (int e = 0; e < VEC; ++e) {
                    run += wt[e];
                    if (wt[e] > 0.f) lp = s0 + k + e;
                    if (yy < 0 && excl + run > rem) yy = s0 + k + e;
                  }
                  if (yy < 0) yy = lp;
                }
                yy = __shfl_sync(kAll, yy, first);
                break;
              }
              base += __shfl_sync(kAll, incl, 31);
            }
            wl = __reduce_max_sync(kAll, wl);
            if (yy < 0) yy = wl;  // the chunk ended before the point by rounding
            if (lane == 0) rr_mail(sh, par, C, rank, make_uint4(static_cast<uint32_t>(yy), 1u, 0u, 0u));
          }
          if (owner != static_cast<int>(rank) && tid == 0)  // an empty message keeps mail C all-to-all
            rr_mail(sh, par, C, rank, make_uint4(0u, 0u, 0u, 0u));
          if (warp == 0) {
            __syncwarp();  // the waiting loop starts converged
            const bool ok = !__any_sync(kAll, !mbar_wait_cluster(&sh.xbar[par], (xk >> 1) & 1u));
            if (lane == 0) {
              sh.y = static_cast<int>(sh.slot[par][owner].x);
              sh.rs = ok ? 0 : SPECDEC_STATUS_TIMEOUT;
            }
          }
          ++xk;
          __syncthreads();
          if (sh.rs) {
            st |= sh.rs;
            break;
          }
          y = sh.y;
        }
      }
      if (child == INT_MAX) break;  // y ends the walk
      if (rank == 0 && tid == 0) {
        P.out_tokens[static_cast<int64_t>(b) * (D + 1) + d] = __ldg(toks + child);
        P.out_path[static_cast<int64_t>(b) * D + d] = child;
      }
      node = child;
      ++d;
    }
  }

  if (rank == 0) {
    const bool err = (st & SPECDEC_STATUS_ERROR_MASK) != 0;
    int32_t* out_t = P.out_tokens + static_cast<int64_t>(b) * (D + 1);
    int32_t* out_p = P.out_path + static_cast<int64_t>(b) * D;
    __syncthreads();  // thread 0's writes of the accepted tokens come first
    for (int i = tid; i <= D; i += NT)
      out_t[i] = err ? -1 : (i < d ? out_t[i] : (i == d ? y : -1));
    for (int i = tid; i < D; i += NT)
      if (err || i >= d) out_p[i] = -1;
    if (tid == 0) {
      P.out_J[b] = err ? -1 : d;
      if (P.out_status) P.out_status[b] = err ? (st & SPECDEC_STATUS_ERROR_MASK) : st;
    }
  }
  // A copy still in flight (a wait gave up) lands before the CTA leaves, and no CTA leaves
  // while a member may still send to it (only possible after a wait gave up).
  if (pending && tid == 0) mbar_wait(&sh.sbar, sphase);
  cluster_arrive_relaxed();
  cluster_wait();
}

constexpr int64_t kRRSliceMaxBytes = 96 * 1024;  // a CTA's logits and q slices
constexpr int kRRTargetCtas = 128;

// Elements per slice for cluster size C (whole 16-byte vectors of both rows), or 0 when C
// does not fit: every CTA must get a non-empty slice whose logits and q fit its stage.
int64_t rr_slice(int V, int es, int C) {
  const int64_t unit = 16 / es;
  const int64_t slice = ((static_cast<int64_t>(V) + C - 1) / C + unit - 1) / unit * unit;
  if (static_cast<int64_t>(C - 1) * slice >= V) return 0;
  if ((slice * es + 15) / 16 * 16 + slice * 4 > kRRSliceMaxBytes) return 0;
  return slice;
}

template <typename T>
cudaError_t launch_rr_cluster_t(const TreeParams& P, int C, int slice, cudaStream_t stream) {
  static unsigned long long configured = 0;
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured & bit)) {
    if (cudaError_t e = cudaFuncSetAttribute(tree_rr_cluster_kernel<T, kTreeThreads>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kRRSliceMaxBytes));
        e != cudaSuccess)
      return e;
    configured |= bit;
  }
  const int qoff = static_cast<int>((static_cast<int64_t>(slice) * static_cast<int64_t>(sizeof(T)) + 15) / 16 * 16);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(P.B) * static_cast<unsigned>(C));
  cfg.blockDim = dim3(kTreeThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(qoff) + static_cast<size_t>(slice) * 4u;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tree_rr_cluster_kernel<T, kTreeThreads>, P, slice, qoff);
}

}  // namespace

int tree_rr_cluster_size(int B, int V, specdec_dtype ldt) {
  const int es = ldt == SPECDEC_BF16 ? 2 : 4;
  if (const int C = test_hook(SPECDEC_HOOK_TREE_CLUSTER)) {  // a fixed size (test hook)
    if ((C == 1 || C == 2 || C == 4 || C == 8) && rr_slice(V, es, C) > 0) return C;
  }
  int best = 0;
  for (int C = 1; C <= kRRMaxC; C *= 2) {
    if (rr_slice(V, es, C) == 0) {
      if (best) break;  // slices would be empty from here on
      continue;         // the rows do not fit yet
    }
    best = C;
    if (static_cast<int64_t>(B) * C >= kRRTargetCtas) break;
  }
  return best;
}

cudaError_t launch_tree_rr_cluster(const TreeParams& P, specdec_dtype ldt, int C, cudaStream_t stream) {
  const int es = ldt == SPECDEC_BF16 ? 2 : 4;
  const int64_t slice = rr_slice(P.V, es, C);
  if (slice <= 0) return cudaErrorInvalidValue;
  if (ldt == SPECDEC_BF16) return launch_rr_cluster_t<uint16_t>(P, C, static_cast<int>(slice), stream);
  return launch_rr_cluster_t<float>(P, C, static_cast<int>(slice), stream);
}

}  // namespace specdec
