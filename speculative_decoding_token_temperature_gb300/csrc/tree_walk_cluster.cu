// The Medusa candidate-tree walk with each row split across a thread-block cluster.
//
// Walk (Medusa notes, section "Attention Tree"): at the current node, sample the target's
// token from softmax(l / T) of that node's logits row (its argmax when greedy); if a child
// of the node carries the token (lowest node index on duplicates) the walk descends, else
// the token ends the walk.  The walk is a chain of dependent row visits, so its time is
// the latency of one visit times the rows visited.  A cluster of C CTAs (C in 1, 2, 4, 8)
// serves one sequence: CTA r stages the contiguous slice [r * slice, (r + 1) * slice) of
// every visited row in its shared memory with bulk copies, and per row
//   slice    its maximum and lowest index (a 64-bit order key) and, sampled, its mass
//            sum 2^((l - m_t) c) relative to each thread's maximum m_t, combined over
//            warps by rescaling to the warp maximum                           -> mail A
//   decide   from every slice's key (and mass, rescaled to the row maximum m): the row's
//            status, the greedy argmax, or the slice and warp chunk holding u * S
//   draw     (sampled) the warp owning u * S scans its chunk in index order; the token
//            goes to every CTA                                                  -> mail C
// Mail is a 16-byte message from every CTA pushed into every member's shared memory
// with st.async, completing transaction bytes on the receiver's mbarrier (no cluster-wide
// barrier per exchange).  Every exchange is all-to-all (in mail C the CTAs that did not
// draw send an empty message), and two mailbox parities alternate: a CTA sends into a
// parity only after it received every member's message of the exchange in between, which
// each member sends only after it received and read the parity's previous messages.
// Every CTA reaches the same decisions from the same messages, so the walk stays uniform
// across the cluster.  Masses are fp32 throughout (fp64 arithmetic is slow on this part
// and this path is a chain of dependent steps): a prefix carries at most a few dozen
// roundings, a relative error of a few 1e-6 at worst, below the 1e-5 band in which a
// draw's boundary is treated as a tie.  Waiting lanes enter their polling loop converged (a warp
// whose lanes wait while another lane still has to send was measured to stall for
// microseconds).  The inputs (tree, tokens, temperature, uniforms) are validated in the
// background of the walk and the walk's result is discarded when they fail, so validation
// loads do not delay the first row; trees of up to kWalkWarpSearch nodes are copied to
// shared memory for the child searches.
// Within a slice each warp owns a contiguous chunk, read by its lanes as consecutive
// 16-byte vectors; index order inside a chunk is (iteration, lane, element).

#include <climits>

#include "specdec_device.cuh"
#include "specdec_internal.h"

namespace specdec {

namespace {

constexpr int kWalkCopy = 32768;      // bytes per bulk copy
constexpr int kWalkMaxCluster = 8;
constexpr int kWalkWarpSearch = 512;  // trees up to this many nodes: one warp finds the child
constexpr unsigned kFull = 0xffffffffu;

// Inclusive prefix over lanes 0..width-1 in lane order (a fixed tree of fp32 adds; width a
// power of two, lanes at or above it keep their own value).
__device__ __forceinline__ float lane_scan(float x, int lane, int width) {
  for (int o = 1; o < width; o <<= 1) {
    const float n = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += n;
  }
  return x;
}

template <typename T>
__device__ __forceinline__ void stage_vec(const T* p, int k, float (&v)[16 / sizeof(T)]) {
  if constexpr (sizeof(T) == 2) {
    const uint4 w = *reinterpret_cast<const uint4*>(p + k);
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
  } else {
    const float4 w = *reinterpret_cast<const float4*>(p + k);
    v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
  }
}

struct WalkShared {
  uint4 slot[2][kWalkMaxCluster];  // mailbox: one 16-byte message per member, by parity
  uint64_t xbar[2];                // mailbox barriers, by parity
  uint64_t sbar;                   // stage barrier
  unsigned long long key[32];      // pass 1: per-warp keys
  float wsum[32];                  // sampled: per-warp masses relative to the warp maximum
  int wlast[32];                   // sampled: per-warp largest index of a finite logit
  float u[kMaxTreeDepth + 1];      // this sequence's uniforms
  int2 tree[kWalkWarpSearch];      // (parent, token) of every node, when N <= kWalkWarpSearch
  float target, wbase;             // the inverse-CDF point; mass before the owner warp's chunk
  float m;                         // row maximum
  int z, owner, ow, lastg, next, y;
  int rs_a, rs_b, rs_y;             // row status after mail A, mail B and the draw
};

// One thread: this CTA's 16-byte message to every member, arming the local barrier for
// all of them.
__device__ __forceinline__ void mail_send(WalkShared& sh, int par, uint32_t C, uint32_t rank, uint4 msg) {
  mbar_expect_tx(&sh.xbar[par], C * 16u);
  const uint32_t sa = smem_addr(&sh.slot[par][rank]);
  const uint32_t ba = smem_addr(&sh.xbar[par]);
  const float4 w = make_float4(__uint_as_float(msg.x), __uint_as_float(msg.y), __uint_as_float(msg.z),
                               __uint_as_float(msg.w));
  for (uint32_t r = 0; r < C; ++r) st_async_16(cluster_map(sa, r), w, cluster_map(ba, r));
}

// Warp: the lowest-index child of `node` carrying token y (INT_MAX: none), from the
// (parent, token) pairs held in shared memory.
__device__ __forceinline__ int warp_find_child(const int2* tree, int N, int node, int y, int lane) {
  int child = INT_MAX;
  for (int j = lane; j < N; j += 32) {
    const int2 pt = tree[j];
    if (pt.x == node && pt.y == y) child = min(child, j);
  }
  return __reduce_min_sync(kFull, child);
}

template <typename T, int NT>
__global__ void __launch_bounds__(NT, 2) tree_walk_cluster_kernel(const TreeParams P, int slice) {
  constexpr int VEC = 16 / static_cast<int>(sizeof(T));
  constexpr int WARPS = NT / 32;
  constexpr int SPAN = 32 * VEC;  // elements per warp iteration
  static_assert(WARPS <= 32 && (WARPS & (WARPS - 1)) == 0, "a power-of-two warp count, one lane per warp");
  extern __shared__ __align__(128) unsigned char stage_raw[];
  __shared__ WalkShared sh;
  __shared__ int sh_i[32];
  const T* stage = reinterpret_cast<const T*>(stage_raw);
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
  const float* ub = P.u + static_cast<int64_t>(b) * (D + 1);
  const bool warp_search = N <= kWalkWarpSearch;
  const uint32_t slice_bytes = static_cast<uint32_t>(n) * static_cast<uint32_t>(sizeof(T));
  auto issue_slice = [=](int node) {  // one thread: this CTA's slice of a node's row (-1: root)
    fence_proxy_async_smem();
    mbar_expect_tx(&sh.sbar, slice_bytes);
    const char* src = reinterpret_cast<const char*>(
        static_cast<const T*>(P.logits) + (static_cast<int64_t>(b) * (N + 1) + (node < 0 ? 0 : 1 + node)) * V + s0);
    for (uint32_t o = 0; o < slice_bytes; o += kWalkCopy)
      bulk_copy_g2s(stage_raw + o, src + o, min(static_cast<uint32_t>(kWalkCopy), slice_bytes - o), &sh.sbar);
  };
  if (tid == 0) {
    mbar_init(&sh.sbar, 1);
    mbar_init(&sh.xbar[0], 1);
    mbar_init(&sh.xbar[1], 1);
    mbar_fence_init();
    issue_slice(-1);  // the root row is read by every walk
  }
  cluster_arrive_relaxed();  // the barriers exist for the other members once all arrived
  bool pending = true;       // (thread 0) a copy into the stage has not been waited for
  uint32_t sphase = 0;       // stage barrier phase
  uint32_t xk = 0;           // exchanges so far

  // Validation in the background: the loads are issued now, the verdict taken after the
  // walk.  The walk itself stays in bounds on any input: rows are nodes' own rows, tokens
  // and parents are only compared, and it stops at max_depth.
  int vst = 0;
  for (int j = tid; j < N; j += NT) {
    const int a = __ldg(P.parents + j);
    if (!(a >= -1 && a < j)) vst |= SPECDEC_STATUS_BAD_TREE;
    const int t = __ldg(toks + j);
    if (t < 0 || t >= V) vst |= SPECDEC_STATUS_BAD_TOKEN;
    if (warp_search) sh.tree[j] = make_int2(a, t);
    int x = j, cnt = 0;  // nodes on the root path of j (bounded walk)
    while (x >= 0 && x < N && cnt <= D) { ++cnt; x = __ldg(P.parents + x); }
    if (cnt > D) vst |= SPECDEC_STATUS_BAD_TREE;
  }
  if (!greedy)
    for (int i = tid; i <= D; i += NT) {
      const float uu = __ldg(ub + i);
      sh.u[i] = uu;
      if (!(uu >= 0.f && uu < 1.f)) vst |= SPECDEC_STATUS_BAD_UNIFORM;
    }
  if (tid == 0 && !(Tb - Tb == 0.f)) vst |= SPECDEC_STATUS_BAD_TEMPERATURE;
  cluster_wait();

  int node = -1, d = 0, st_rows = 0;
  for (;;) {
    // ---- the slice: maximum and its lowest index (the order key), and for a sampled row
    // the mass sum 2^((l - m_t) c) relative to each thread's maximum m_t (a second read of
    // the thread's elements in shared memory) ---------------------------------------------
    const bool landed = mbar_wait(&sh.sbar, sphase);
    if (landed) {
      sphase ^= 1u;
      pending = false;
    }
    float best = -kInf, s = 0.f;
    int bidx = INT_MAX, lastf = -1;
    bool nan = false;
    if (landed) {
      for (int k = w0 + lane * VEC; k < w1; k += SPAN) {  // each thread visits its indices in order
        float v[VEC];
        stage_vec<T>(stage, k, v);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          nan |= (v[e] != v[e]);
          if (v[e] > best) { best = v[e]; bidx = s0 + k + e; }
        }
      }
      if (!greedy && best > -kInf)  // the thread's mass relative to its maximum (shared memory again)
        for (int k = w0 + lane * VEC; k < w1; k += SPAN) {
          float v[VEC];
          stage_vec<T>(stage, k, v);
#pragma unroll
          for (int e = 0; e < VEC; ++e)
            if (v[e] > -kInf) {
              s += ex2((v[e] - best) * c);
              lastf = s0 + k + e;
            }
        }
    }
    const unsigned long long wkey = warp_max_key(landed ? order_key(best, bidx, nan) : kKeyTimeout);
    if (!greedy) {  // the warp's mass relative to the warp maximum
      const float wm = key_value(wkey);
      float sw = best > -kInf ? s * ex2((best - wm) * c) : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sw += __shfl_xor_sync(kFull, sw, o);
      lastf = __reduce_max_sync(kFull, lastf);
      if (lane == 0) {
        sh.wsum[warp] = sw;
        sh.wlast[warp] = lastf;
      }
    }
    if (lane == 0) sh.key[warp] = wkey;
    __syncthreads();  // also: every read of the stage but the draw's is done

    // ---- warp 0: the CTA's key (and masses), the exchange, and the row's decision -------
    if (warp == 0) {
      const int par = static_cast<int>(xk & 1u);
      const unsigned long long kw = lane < WARPS ? sh.key[lane] : 0ull;
      const unsigned long long ckey = warp_max_key(kw);
      const float mr = key_value(ckey);  // this slice's maximum
      int lp = -1;
      float pre = 0.f;  // sampled: mass through warp `lane`'s chunk, relative to mr
      float sw = 0.f;
      if (!greedy) {
        const float kv = key_value(kw);
        sw = (lane < WARPS && kv > -kInf) ? sh.wsum[lane] * ex2((kv - mr) * c) : 0.f;
        pre = lane_scan(sw, lane, WARPS);
        lp = __reduce_max_sync(kFull, lane < WARPS ? sh.wlast[lane] : -1);
      }
      const float mass = __shfl_sync(kFull, pre, WARPS - 1);
      if (lane == 0) {
        const uint4 msg = make_uint4(static_cast<uint32_t>(ckey), static_cast<uint32_t>(ckey >> 32),
                                     __float_as_uint(mass), static_cast<uint32_t>(lp));
        mail_send(sh, par, C, rank, msg);
      }
      __syncwarp();
      const bool ok = !__any_sync(kFull, !mbar_wait_cluster(&sh.xbar[par], (xk >> 1) & 1u));
      unsigned long long kr = 0ull;
      float sr = 0.f;
      int lr = -1;
      if (lane < static_cast<int>(C)) {
        const uint4 a = sh.slot[par][lane];
        kr = (static_cast<unsigned long long>(a.y) << 32) | a.x;
        sr = __uint_as_float(a.z);
        lr = static_cast<int>(a.w);
      }
      const unsigned long long K = warp_max_key(kr);
      const float m = key_value(K);
      int rs = 0;
      if (!ok || K == kKeyTimeout) rs = SPECDEC_STATUS_TIMEOUT;
      else if (!(m == m) || m == kInf) rs = SPECDEC_STATUS_BAD_LOGIT;
      else if (m == -kInf) rs = SPECDEC_STATUS_EMPTY_ROW;
      if (rs == 0 && greedy && warp_search) {  // the greedy token is the argmax: descend now
        const int y = key_index(K);
        const int child = warp_find_child(sh.tree, N, node, y, lane);
        if (lane == 0) {
          const bool down = child != INT_MAX && d < D;
          if (rank == 0) {
            P.out_tokens[static_cast<int64_t>(b) * (D + 1) + d] = y;
            if (down) P.out_path[static_cast<int64_t>(b) * D + d] = child;
          }
          sh.next = down ? child : -1;
          if (down) {
            issue_slice(child);
            pending = true;
          }
        }
      }
      if (rs == 0 && !greedy) {
        // every slice's mass scaled to the row maximum; the slice, then the warp chunk,
        // that holds the inverse-CDF point u * S
        lr = __reduce_max_sync(kFull, lr);
        const float mk = key_value(kr);
        const float f = (lane < static_cast<int>(C) && mk > -kInf) ? ex2((mk - m) * c) : 0.f;
        const float incl = lane_scan(sr * f, lane, static_cast<int>(C));  // mass through slice `lane`
        const float target = __shfl_sync(kFull, incl, static_cast<int>(C) - 1) * sh.u[d];
        const unsigned hit = __ballot_sync(kFull, lane < static_cast<int>(C) && incl > target);
        const int owner = hit ? __ffs(hit) - 1 : -1;
        const float before = __shfl_sync(kFull, incl, owner > 0 ? owner - 1 : 0);
        const float obase = owner > 0 ? before : 0.f;
        int ow = -1;
        float wb = 0.f;
        if (owner == static_cast<int>(rank)) {
          const float fme = ex2((mr - m) * c);
          const unsigned h2 = __ballot_sync(kFull, lane < WARPS && obase + pre * fme > target);
          const unsigned pos = __ballot_sync(kFull, lane < WARPS && sw > 0.f);
          ow = h2 ? __ffs(h2) - 1 : (pos ? 31 - __clz(pos) : 0);  // past the end only by rounding
          const float prev = __shfl_sync(kFull, pre, ow > 0 ? ow - 1 : 0);
          wb = ow > 0 ? obase + prev * fme : obase;
        }
        if (lane == 0) {
          sh.owner = owner;
          sh.ow = ow;
          sh.lastg = lr;
          sh.target = target;
          sh.wbase = wb;
        }
      }
      if (lane == 0) {
        sh.rs_a = rs;
        sh.m = m;
        sh.z = key_index(K);
      }
    }
    ++xk;
    __syncthreads();
    if (sh.rs_a) {
      st_rows |= sh.rs_a;
      break;
    }
    if (greedy && warp_search) {
      if (sh.next < 0) break;
      node = sh.next;
      ++d;
      continue;
    }

    int y = sh.z;  // greedy: the argmax
    int ry = 0;    // a time-out while drawing
    if (!greedy) {
      // ---- draw: the owner warp scans its chunk in index order; mail C ---------------
      const float m = sh.m;
      const int owner = sh.owner;
      const int par = static_cast<int>(xk & 1u);
      if (owner == static_cast<int>(rank) && warp == sh.ow) {
        const float target = sh.target;
        float base = sh.wbase;
        int yy = -1, wl = -1;
        for (int k0 = w0; k0 < w1; k0 += SPAN) {
          const int k = k0 + lane * VEC;
          float wt[VEC];
          float a = 0.f;
          if (k < w1) {
            float v[VEC];
            stage_vec<T>(stage, k, v);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
              wt[e] = ex2((v[e] - m) * c);
              a += wt[e];
              if (wt[e] > 0.f) wl = s0 + k + e;
            }
          } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) wt[e] = 0.f;
          }
          float incl = a;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += t;
          }
          const float rem = target - base;  // mass still to pass at this tile's start
          const unsigned hit = __ballot_sync(kFull, incl > rem);
          if (hit) {
            const int first = __ffs(hit) - 1;
            if (lane == first) {
              const float excl = incl - a;
              float run = 0.f;
              int lpos = -1;
#pragma unroll
              for (int e = 0; e < VEC; ++e) {
                run += wt[e];
                if (wt[e] > 0.f) lpos = s0 + k + e;
                if (yy < 0 && excl + run > rem) yy = s0 + k + e;
              }
              if (yy < 0) yy = lpos;
            }
            yy = __shfl_sync(kFull, yy, first);
            break;
          }
          base += __shfl_sync(kFull, incl, 31);
        }
        wl = __reduce_max_sync(kFull, wl);
        if (yy < 0) yy = wl;  // the chunk ended before the point by rounding
        if (yy < 0) yy = sh.lastg;
        if (lane == 0) {
          const uint4 msg = make_uint4(static_cast<uint32_t>(yy), 1u, 0u, 0u);
          mail_send(sh, par, C, rank, msg);
        }
      }
      if (owner != static_cast<int>(rank) && tid == 0) {  // an empty message keeps mail C all-to-all
        const uint4 msg = make_uint4(0u, 0u, 0u, 0u);
        mail_send(sh, par, C, rank, msg);
      }
      if (warp == 0) {
        __syncwarp();  // the waiting loop starts converged
        const bool ok = !__any_sync(kFull, !mbar_wait_cluster(&sh.xbar[par], (xk >> 1) & 1u));
        if (!ok) ry = SPECDEC_STATUS_TIMEOUT;
        else y = (owner >= 0) ? static_cast<int>(sh.slot[par][owner].x) : sh.lastg;
      }
      ++xk;
    }

    // ---- descend into the lowest-index child carrying y (the same in every CTA) --------
    int child = -1;
    if (warp_search) {
      if (warp == 0) {
        const int ch = ry ? INT_MAX : warp_find_child(sh.tree, N, node, y, lane);
        const bool down = !ry && ch != INT_MAX && d < D;
        if (lane == 0) {
          if (!ry && rank == 0) {
            P.out_tokens[static_cast<int64_t>(b) * (D + 1) + d] = y;
            if (down) P.out_path[static_cast<int64_t>(b) * D + d] = ch;
          }
          sh.rs_y = ry;
          sh.next = down ? ch : -1;
          if (down) {
            issue_slice(ch);
            pending = true;
          }
        }
      }
      __syncthreads();
      if (sh.rs_y) {
        st_rows |= sh.rs_y;
        break;
      }
      child = sh.next;
    } else {
      if (tid == 0) {
        sh.rs_y = ry;
        sh.y = y;
      }
      __syncthreads();
      if (sh.rs_y) {
        st_rows |= sh.rs_y;
        break;
      }
      y = sh.y;
      int ch = INT_MAX;
      for (int j = tid; j < N; j += NT)
        if (__ldg(P.parents + j) == node && __ldg(toks + j) == y) ch = min(ch, j);
      ch = Block<NT>::min_int(ch, sh_i);
      const bool down = ch != INT_MAX && d < D;
      if (tid == 0) {
        if (rank == 0) {
          P.out_tokens[static_cast<int64_t>(b) * (D + 1) + d] = y;
          if (down) P.out_path[static_cast<int64_t>(b) * D + d] = ch;
        }
        if (down) {
          issue_slice(ch);
          pending = true;
        }
      }
      child = down ? ch : -1;
    }
    if (child < 0) break;
    node = child;
    ++d;
  }

  // The verdict of validation; a failed input discards the walk.
  vst = Block<NT>::or_int(vst, sh_i);
  const int st = (vst & SPECDEC_STATUS_ERROR_MASK) ? vst : (vst | st_rows);
  if (rank == 0) {
    const bool err = (st & SPECDEC_STATUS_ERROR_MASK) != 0;
    int32_t* out_t = P.out_tokens + static_cast<int64_t>(b) * (D + 1);
    int32_t* out_p = P.out_path + static_cast<int64_t>(b) * D;
    for (int i = tid; i <= D; i += NT)
      if (err || i > d) out_t[i] = -1;
    for (int i = tid; i < D; i += NT)
      if (err || i >= d) out_p[i] = -1;
    if (tid == 0) {
      P.out_J[b] = err ? -1 : d;
      if (P.out_status) P.out_status[b] = st;
    }
  }
  // A copy still in flight (a wait gave up) lands before the CTA leaves, and no CTA leaves
  // while a member may still send to it (only possible after a wait gave up).
  if (pending && tid == 0) mbar_wait(&sh.sbar, sphase);
  cluster_arrive_relaxed();
  cluster_wait();
}

constexpr int64_t kWalkSliceMaxBytes = 96 * 1024;  // a slice of a row staged per CTA
constexpr int kWalkTargetCtas = 128;               // clusters grow until B * C reaches this

// Elements per slice for cluster size C (whole 16-byte vectors), or 0 when C does not fit:
// every CTA must get a non-empty slice that fits its stage.
int64_t walk_slice(int V, int es, int C) {
  const int64_t unit = 16 / es;
  const int64_t slice = ((static_cast<int64_t>(V) + C - 1) / C + unit - 1) / unit * unit;
  if (static_cast<int64_t>(C - 1) * slice >= V) return 0;
  if (slice * es > kWalkSliceMaxBytes) return 0;
  return slice;
}

template <typename T>
cudaError_t launch_cluster_t(const TreeParams& P, int C, int slice, cudaStream_t stream) {
  static unsigned long long configured = 0;
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured & bit)) {
    if (cudaError_t e = cudaFuncSetAttribute(tree_walk_cluster_kernel<T, kTreeThreads>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kWalkSliceMaxBytes));
        e != cudaSuccess)
      return e;
    configured |= bit;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(P.B) * static_cast<unsigned>(C));
  cfg.blockDim = dim3(kTreeThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(slice) * sizeof(T);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tree_walk_cluster_kernel<T, kTreeThreads>, P, slice);
}

}  // namespace

int tree_walk_cluster_size(int B, int V, specdec_dtype ldt) {
  const int es = ldt == SPECDEC_BF16 ? 2 : 4;
  if (const int C = test_hook(SPECDEC_HOOK_TREE_CLUSTER)) {  // a fixed size (test hook)
    if ((C == 1 || C == 2 || C == 4 || C == 8) && walk_slice(V, es, C) > 0) return C;
  }
  int best = 0;
  for (int C = 1; C <= kWalkMaxCluster; C *= 2) {
    if (walk_slice(V, es, C) == 0) {
      if (best) break;  // slices would be empty from here on
      continue;         // the row does not fit yet
    }
    best = C;
    if (static_cast<int64_t>(B) * C >= kWalkTargetCtas) break;
  }
  return best;
}

cudaError_t launch_tree_walk_cluster(const TreeParams& P, specdec_dtype ldt, int C, cudaStream_t stream) {
  const int es = ldt == SPECDEC_BF16 ? 2 : 4;
  const int64_t slice = walk_slice(P.V, es, C);
  if (slice <= 0 || P.D > kMaxTreeDepth) return cudaErrorInvalidValue;
  if (ldt == SPECDEC_BF16) return launch_cluster_t<uint16_t>(P, C, static_cast<int>(slice), stream);
  return launch_cluster_t<float>(P, C, static_cast<int>(slice), stream);
}

}  // namespace specdec
