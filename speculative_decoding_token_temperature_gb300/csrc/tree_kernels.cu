// Token-tree kernels: the Medusa candidate-tree walk and the tree-attention mask.
//
// Walk (Medusa notes, section "Attention Tree"): one CTA per sequence.  At the current
// node the CTA makes one pass over that node's logits row for the maximum and its lowest
// index; a greedy sequence takes the argmax, a sampled one makes a second pass for the
// total mass of 2^((l - max) * log2(e) / T) and scans the row in index order for the
// smallest k with C_k > u_d * S (inverse CDF of softmax(l / T)).  If a child of the node
// carries the drawn token (lowest node index on duplicates) the walk descends; otherwise
// the drawn token ends the walk.  Only the rows on the walk are read.  This one-CTA walk
// over global memory serves rows that are not 16-byte aligned or too long to stage; the
// others take the cluster walk of tree_walk_cluster.cu.
//
// Mask (SD 20.5, box "Token tree and tree attention"): node i sees every prefix column,
// itself and its ancestors; position id P + depth(i).

#include <climits>

#include "specdec_device.cuh"
#include "specdec_internal.h"

namespace specdec {

namespace {

template <typename T, int VEC, int NT>
__global__ void __launch_bounds__(NT) tree_walk_kernel(const TreeParams P) {
  __shared__ float sh_f[32];
  __shared__ int sh_i[32];
  __shared__ double sh_d[32];
  __shared__ int s_y;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int N = P.N, V = P.V, D = P.D;
  const float Tb = __ldg(P.temps + b);
  const bool greedy = !(Tb >= SPECDEC_GREEDY_TEMPERATURE);
  const float c = greedy ? 0.f : kLog2e / Tb;
  const int32_t* toks = P.node_tokens + static_cast<int64_t>(b) * N;
  int32_t* out_t = P.out_tokens + static_cast<int64_t>(b) * (D + 1);
  int32_t* out_p = P.out_path + static_cast<int64_t>(b) * D;

  // Validate the tree, the tokens, the temperature and the uniforms.
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
    for (int d = tid; d <= D; d += NT) {
      const float uu = __ldg(P.u + static_cast<int64_t>(b) * (D + 1) + d);
      if (!(uu >= 0.f && uu < 1.f)) bu = SPECDEC_STATUS_BAD_UNIFORM;
    }
    st |= bu;
  }
  st = Block<NT>::or_int(st, sh_i);

  int node = -1, d = 0;
  if (!(st & SPECDEC_STATUS_ERROR_MASK)) {
    for (;;) {
      const int row = (node < 0) ? 0 : 1 + node;
      const T* lrow = static_cast<const T*>(P.logits) + (static_cast<int64_t>(b) * (N + 1) + row) * V;
      // pass 1: maximum and its lowest index (each thread walks its vectors in index order)
      float best = -kInf;
      int bidx = INT_MAX;
      bool nan = false;
      for (int k = tid * VEC; k < V; k += NT * VEC) {
        float v[VEC];
        VecLoad<T, VEC>::load(lrow, k, v);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          nan |= (v[e] != v[e]);
          if (v[e] > best) { best = v[e]; bidx = k + e; }  // strict: first index kept on ties
        }
      }
      if (nan) best = __int_as_float(0x7fc00000);
      const float m = Block<NT>::max(best, sh_f);
      int cand = (best == m) ? bidx : INT_MAX;
      const int z = Block<NT>::min_int(cand, sh_i);
      int rs = 0;
      if (!(m == m) || m == kInf) rs = SPECDEC_STATUS_BAD_LOGIT;
      else if (m == -kInf) rs = SPECDEC_STATUS_EMPTY_ROW;
      if (rs) { st |= rs; break; }

      int y = z;
      if (!greedy) {
        // pass 2: total mass (fp32 within a thread and a warp, fp64 across warps)
        float tot = 0.f;
        for (int k = tid * VEC; k < V; k += NT * VEC) {
          float v[VEC];
          VecLoad<T, VEC>::load(lrow, k, v);
          float a = 0.f;
#pragma unroll
          for (int e = 0; e < VEC; ++e) a += ex2((v[e] - m) * c);
          tot += a;
        }
        const double S = Block<NT>::sum_f(tot, sh_d);
        const double target = static_cast<double>(__ldg(P.u + static_cast<int64_t>(b) * (D + 1) + d)) * S;
        // pass 3: tiles of NT vectors in index order until the running mass passes target
        double base = 0.0;
        if (tid == 0) s_y = -1;
        int last_pos = -1;
        for (int k0 = 0; k0 < V; k0 += NT * VEC) {
          const int k = k0 + tid * VEC;
          float w[VEC];
          float a = 0.f;
          if (k < V) {
            float v[VEC];
            VecLoad<T, VEC>::load(lrow, k, v);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
              w[e] = ex2((v[e] - m) * c);
              a += w[e];
              if (w[e] > 0.f) last_pos = k + e;
            }
          } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) w[e] = 0.f;
          }
          double total;
          const double incl = Block<NT>::inclusive_scan_f(a, sh_d, total);
          if (base + total > target) {
            const int first = Block<NT>::min_int((base + incl > target) ? tid : INT_MAX, sh_i);
            if (tid == first) {
              const double excl = base + (incl - static_cast<double>(a));
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
          base += total;
        }
        __syncthreads();
        y = s_y;
        if (y < 0) y = -Block<NT>::min_int(last_pos < 0 ? INT_MAX : -last_pos, sh_i);
      }

      // descend into the lowest-index child carrying y, if any
      int child = INT_MAX;
      for (int j = tid; j < N; j += NT)
        if (__ldg(P.parents + j) == node && __ldg(toks + j) == y) child = min(child, j);
      child = Block<NT>::min_int(child, sh_i);
      if (tid == 0) out_t[d] = y;
      if (child == INT_MAX) break;
      if (tid == 0) out_p[d] = child;
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
    if (P.out_status) P.out_status[b] = st;
  }
}

template <typename T, int VEC>
cudaError_t launch_walk_t(const TreeParams& P, cudaStream_t stream) {
  return launch_kernel(tree_walk_kernel<T, VEC, kTreeThreads>, dim3(P.B), dim3(kTreeThreads), 0, stream, 0, P);
}

// Bytes 0..n-1 of a little-endian 8-byte word set to 1 (0 <= n <= 8).
__device__ __forceinline__ unsigned long long mask_ones(int n) {
  return n >= 8 ? 0x0101010101010101ull : (0x0101010101010101ull & ((1ull << (8 * n)) - 1ull));
}

// One warp per node, i.e. per mask row: the row is written as 16-byte words (prefix columns
// 1, node columns 0; the row's unaligned ends byte by byte), then the warp's first lane
// walks the node's ancestor chain once, setting the node's own column and each ancestor's
// to 1 and counting the depth.  A row costs one pass of coalesced stores plus depth + 1
// byte stores, instead of an ancestor walk per byte.
constexpr int kMaskWarps = 8;
__global__ void __launch_bounds__(kMaskWarps * 32) tree_mask_kernel(const int32_t* __restrict__ parents, int N,
                                                                   int P, uint8_t* __restrict__ mask,
                                                                   int64_t* __restrict__ pos,
                                                                   int32_t* __restrict__ depth,
                                                                   int32_t* __restrict__ status) {
  __shared__ int sh_i[32];
  const int lane = threadIdx.x & 31;
  const int64_t W = static_cast<int64_t>(P) + N;
  const int nwarps = static_cast<int>(gridDim.x) * kMaskWarps;
  for (int i = static_cast<int>(blockIdx.x) * kMaskWarps + static_cast<int>(threadIdx.x >> 5); i < N; i += nwarps) {
    uint8_t* row = mask + static_cast<int64_t>(i) * W;
    const int64_t head = min(W, static_cast<int64_t>((16u - (reinterpret_cast<uintptr_t>(row) & 15u)) & 15u));
    const int64_t nvec = (W - head) / 16;
    const int64_t tail = head + nvec * 16;
    for (int64_t c = lane; c < head; c += 32) row[c] = c < P ? 1 : 0;
    uint4* vrow = reinterpret_cast<uint4*>(row + head);
    for (int64_t k = lane; k < nvec; k += 32) {
      const int64_t c0 = head + 16 * k;  // the word's first column
      const int n1 = static_cast<int>(min(static_cast<int64_t>(16), max(static_cast<int64_t>(0), P - c0)));
      const unsigned long long lo = mask_ones(min(n1, 8)), hi = mask_ones(max(n1 - 8, 0));
      vrow[k] = make_uint4(static_cast<uint32_t>(lo), static_cast<uint32_t>(lo >> 32), static_cast<uint32_t>(hi),
                           static_cast<uint32_t>(hi >> 32));
    }
    for (int64_t c = tail + lane; c < W; c += 32) row[c] = c < P ? 1 : 0;
    __syncwarp();  // (orders the words before the ancestor bytes written over them)
    if (lane == 0) {
      // the chain climbs strictly (parents[a] < a), so it ends within N steps even for a
      // bad tree (whose outputs are unspecified; its status says so)
      int a = i, d = 0, pa = __ldg(parents + i);
      row[P + i] = 1;
      while (pa >= 0 && pa < a) {
        row[P + pa] = 1;
        a = pa;
        pa = __ldg(parents + a);
        ++d;
      }
      pos[i] = static_cast<int64_t>(P) + d;
      if (depth) depth[i] = d;
    }
  }
  if (blockIdx.x == 0) {
    int bad = 0;
    for (int i = threadIdx.x; i < N; i += blockDim.x) {
      const int pa = __ldg(parents + i);
      if (!(pa >= -1 && pa < i)) bad = SPECDEC_STATUS_BAD_TREE;
    }
    bad = Block<kMaskWarps * 32>::or_int(bad, sh_i);
    if (threadIdx.x == 0) *status = bad;
  }
}

}  // namespace

cudaError_t launch_tree_walk(const TreeParams& P, specdec_dtype ldt, bool vector_path,
                             cudaStream_t stream) {
  if (vector_path) {
    if (const int C = tree_walk_cluster_size(P.B, P.V, ldt); C > 0)
      return launch_tree_walk_cluster(P, ldt, C, stream);
    if (ldt == SPECDEC_BF16) return launch_walk_t<uint16_t, 8>(P, stream);
    return launch_walk_t<float, 4>(P, stream);
  }
  if (ldt == SPECDEC_BF16) return launch_walk_t<uint16_t, 1>(P, stream);
  return launch_walk_t<float, 1>(P, stream);
}

cudaError_t launch_tree_mask(const int32_t* parents, int N, int prefix_len, uint8_t* mask,
                             int64_t* pos, int32_t* depth, int32_t* status, cudaStream_t stream) {
  // one warp per row, at most eight 256-thread blocks per SM at once
  int64_t blocks = (static_cast<int64_t>(N) + kMaskWarps - 1) / kMaskWarps;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_kernel(tree_mask_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kMaskWarps * 32), 0, stream, 0,
                       parents, N, prefix_len, mask, pos, depth, status);
}

}  // namespace specdec
