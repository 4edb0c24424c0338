// Streaming chain verification for 16-byte aligned rows (the common case).
//
// Four kernels chained with programmatic dependent launch; each kernel boundary orders
// one phase's results before the next, so no kernel needs an in-flight fence:
//
//   stats   persistent, one CTA per SM; every warp is an independent pipeline holding
//           three 1-D bulk copies (cp.async.bulk completed on an mbarrier) of its next
//           work items in shared memory.  Item = (row, 4 KB chunk) of logits.  Per chunk:
//           maximum (packed max.NaN.bf16x2 for bf16), then for sampled sequences the sum
//           of 2^((l - m) * log2(e) / T) (packed f32x2 arithmetic, one ex2 per element), or
//           for greedy sequences the lowest index of the maximum.
//   decide  one CTA per sequence: merges every row's chunk summaries in a fixed order,
//           runs the accept tests in order (SD 20.5, "A round of speculative sampling":
//           accept x_i iff u_i * q_i(x_i) < p_i(x_i); J = leading accepts; greedy rows
//           accept iff x_i == argmax, "A round of greedy speculative decoding"), writes the
//           accepted prefix and lists the sequences that draw an extra token.
//   draw    persistent like stats.  Item = (listed sequence, 1024-element chunk) of its
//           drawn row: residual weights (p_J - q_J)+ (q == 0 for the bonus row; SD 20.5,
//           "The speculative sampling rule", "Speculative verification in PyTorch") and
//           their chunk mass.
//   finish  one warp per sequence: locates the chunk whose running mass passes u * S and
//           scans it in index order for the smallest k with C_k > u * S.

#include "stream_common.cuh"

namespace specdec {

namespace {

#ifndef SPECDEC_DRAW_LIST_CACHE
#define SPECDEC_DRAW_LIST_CACHE 256
#endif
constexpr int kDrawListCache = SPECDEC_DRAW_LIST_CACHE;  // draw-list entries kept in shared memory
constexpr int kDecideThreads = 256;

// ---------------------------------------------------------------------------------
// stats
// ---------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kStatsWarps * 32, 1) chain_stats_stream_kernel(const ChainParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t bars[kStatsWarps][kStatsStages];
  constexpr int VPL = kStatsChunkBytes / 16 / 32;  // 16-byte vectors per lane per chunk
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t NW = gridDim.x * kStatsWarps;
  const uint32_t gw = blockIdx.x * kStatsWarps + warp;
  unsigned char* buf = smem + static_cast<size_t>(warp) * kStatsStages * kStatsChunkBytes;
  uint64_t* bar = bars[warp];
  const uint32_t R = P.gamma + 1;
  const uint32_t nch = P.nch;
  const int64_t row_bytes = static_cast<int64_t>(P.V) * sizeof(T);
  const uint32_t n_items = static_cast<uint32_t>(P.B) * R * nch;  // < 2^31 (checked on the host)
  const char* base = static_cast<const char*>(P.logits);

  if (lane == 0) {
    for (int s = 0; s < kStatsStages; ++s) mbar_init(&bar[s], 1);
    mbar_fence_init();
  }
  __syncwarp();

  auto issue = [&](uint32_t it, int s) {
    const uint32_t row = it / nch;
    const int64_t off = static_cast<int64_t>(it - row * nch) * kStatsChunkBytes;
    const uint32_t bytes = static_cast<uint32_t>(min(static_cast<int64_t>(kStatsChunkBytes), row_bytes - off));
    mbar_expect_tx(&bar[s], bytes);
    bulk_copy_g2s(buf + s * kStatsChunkBytes, base + static_cast<int64_t>(row) * row_bytes + off, bytes, &bar[s]);
  };
  uint32_t issued = 0;
  for (uint32_t it = gw; issued < kStatsStages && it < n_items; it += NW, ++issued)
    if (lane == 0) issue(it, issued);

  uint32_t k = 0;
  for (uint32_t it = gw; it < n_items; it += NW, ++k) {
    const int s = static_cast<int>(k % kStatsStages);
    if (!mbar_wait(&bar[s], (k / kStatsStages) & 1u)) {
      if (lane == 0) drain_after_timeout(bar, kStatsStages, k, issued, P.ws.error);
      break;
    }
    const uint32_t row = it / nch;
    const uint32_t ch = it - row * nch;
    const uint32_t b = row / R;
    const int nv = static_cast<int>(min(static_cast<int64_t>(kStatsChunkBytes),
                                        row_bytes - static_cast<int64_t>(ch) * kStatsChunkBytes) / 16);
    const uint4* vb = reinterpret_cast<const uint4*>(buf + s * kStatsChunkBytes);
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
    // the chunk is in registers: refill this stage with the item kStatsStages steps ahead
    const uint32_t nx = it + kStatsStages * NW;
    const bool refill = nx < n_items && nx > it;
    if (lane == 0 && refill) {
      fence_proxy_async_smem();
      issue(nx, s);
    }
    issued += refill ? 1u : 0u;

    const float Tb = P.greedy_only ? 0.f : __ldg(P.temps + b);
    const bool greedy = P.greedy_only || is_greedy(Tb);
    const float c = greedy ? 0.f : kLog2e / Tb;
    const float4 sum = chunk_summary<T>(w, nv, ch, greedy, c);
    if (lane == 0) P.ws.partials[it] = sum;
  }
}

// ---------------------------------------------------------------------------------
// decide: one CTA per sequence
// ---------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kDecideThreads) chain_decide_kernel(const ChainParams P) {
  __shared__ float s_m[kStreamMaxRows], s_Z[kStreamMaxRows];
  __shared__ int s_z[kStreamMaxRows];
  grid_launch_dependents();
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = P.gamma + 1;
  const int nch = P.nch;
  const float Tb = P.greedy_only ? 0.f : __ldg(P.temps + b);
  const bool greedy = P.greedy_only || is_greedy(Tb);
  const float c = greedy ? 0.f : kLog2e / Tb;

  // Inputs only (drafts, the logit and q at each draft, uniforms): fetched before waiting
  // for the statistics kernel, so these loads overlap its tail.  Lane i < gamma holds
  // position i; lane gamma holds the bonus row and the draw's uniform.
  // Checks of one position, in order: its logits row, then its draft token, then (when
  // sampled) its draft probability and uniform together.
  int x = -1, tok_err = 0, qu_err = 0;
  float lx = 0.f, qx = 0.f, ux = 0.f;
  if (warp == 0) {
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
  grid_dependency_wait();

  // merge each row's chunk summaries (fixed order: deterministic); warps take rows
  for (int r = warp; r < R; r += kDecideThreads / 32) {
    const float4* pp = P.ws.partials + (static_cast<int64_t>(b) * R + r) * nch;
    RowSum acc;
    acc.m = -kInf;
    acc.Z = 0.f;
    acc.z = INT_MAX;
    for (int q = lane; q < nch; q += 32) {
      const float4 f = __ldcg(pp + q);
      RowSum t;
      t.m = f.x;
      t.Z = f.y;
      t.z = __float_as_int(f.z);
      acc = merge(acc, t, c);
    }
    acc = warp_merge(acc, c);
    if (lane == 0) {
      s_m[r] = acc.m;
      s_Z[r] = acc.Z;
      s_z[r] = acc.z;
    }
  }
  __syncthreads();
  if (warp != 0) return;

  // Positions are evaluated left to right and evaluation stops at the first rejection
  // (SD 20.5, "A whole round of speculative sampling"); lane i evaluates position i and
  // the first lane that stops -- by an error or a rejection -- decides the round.
  float m = -kInf, Z = 0.f;
  int z = INT_MAX, warn = 0, row_err = 0;
  if (lane < R) {
    m = s_m[lane];
    Z = s_Z[lane];
    z = s_z[lane];
    if (!(m == m) || m == kInf) row_err = SPECDEC_STATUS_BAD_LOGIT;
    else if (m == -kInf) row_err = SPECDEC_STATUS_EMPTY_ROW;
  }
  const int err = row_err ? row_err : (tok_err ? tok_err : qu_err);
  bool acc = false;
  float px = kNaN;
  if (lane < P.gamma && !err) {
    if (greedy) {
      acc = (x == z);
    } else {
      px = ex2((lx - m) * c) / Z;
      if (qx == 0.f) {
        warn |= SPECDEC_STATUS_ZERO_Q;
        acc = px > 0.f;
      } else {
        acc = ux * qx < px;
      }
    }
  }
  const bool stop = (lane < R) && (err != 0 || lane == P.gamma || !acc);
  const int s_stop = __ffs(__ballot_sync(0xffffffffu, stop)) - 1;  // <= gamma
  int st = __shfl_sync(0xffffffffu, err, s_stop);
  st |= __reduce_or_sync(0xffffffffu, lane <= s_stop ? warn : 0);
  if (!P.greedy_only && !(Tb - Tb == 0.f)) st = SPECDEC_STATUS_BAD_TEMPERATURE;
  const float uG = __shfl_sync(0xffffffffu, ux, P.gamma);
  if (!(st & SPECDEC_STATUS_ERROR_MASK) && !greedy && !(uG >= 0.f && uG < 1.f)) st |= SPECDEC_STATUS_BAD_UNIFORM;
  const bool failed = (st & SPECDEC_STATUS_ERROR_MASK) != 0;
  const int J = failed ? -1 : s_stop;
  if (lane < P.gamma && P.out_p_draft)
    P.out_p_draft[static_cast<int64_t>(b) * P.gamma + lane] = (!failed && lane <= J) ? px : kNaN;
  const int zJ = __shfl_sync(0xffffffffu, z, s_stop);
  const float mJ = __shfl_sync(0xffffffffu, m, s_stop);
  const float ZJ = __shfl_sync(0xffffffffu, Z, s_stop);
  if (lane < R) {
    int tok = -1;
    if (J >= 0) {
      if (lane < J) tok = x;
      else if (lane == J && greedy) tok = zJ;
    }
    P.out_tokens[static_cast<int64_t>(b) * R + lane] = tok;
  }
  if (lane == 0) {
    P.out_J[b] = J;
    if (P.out_status) P.out_status[b] = st;
    const bool draw = (J >= 0) && !greedy;
    SeqState sq;
    sq.meta = make_int4(J, draw ? 1 : 0, st, 0);
    sq.row = make_float4(draw ? mJ : 0.f, draw ? ZJ : 0.f, c, draw ? uG : 0.f);
    P.ws.seq[b] = sq;
    if (draw) {
      DrawEntry d;
      d.loc = make_int4(b, J, b, 0);  // (sequence, drawn row, mass slot, 0)
      d.row = make_float4(mJ, c, 1.f / ZJ, 0.f);
      P.ws.draw_list[atomicAdd(P.ws.draw_count, 1u)] = d;
    }
  }
}

// ---------------------------------------------------------------------------------
// draw
// ---------------------------------------------------------------------------------

template <typename T>
constexpr int draw_stages() { return sizeof(T) == 2 ? kDrawStages : kDrawStagesF32; }

template <typename T>
constexpr int draw_smem_bytes() {
  return kDrawWarps * draw_stages<T>() * (kDrawChunk * static_cast<int>(sizeof(T)) + kDrawChunk * 4) +
         kDrawListCache * static_cast<int>(sizeof(DrawEntry));
}
static_assert(draw_smem_bytes<uint16_t>() <= 227 * 1024, "bf16 draw stages exceed shared memory");
static_assert(draw_smem_bytes<float>() <= 227 * 1024, "fp32 draw stages exceed shared memory");
static_assert(kStatsWarps * kStatsStages * kStatsChunkBytes <= 227 * 1024, "statistics stages exceed shared memory");

template <typename T>
__global__ void __launch_bounds__(kDrawWarps * 32, 1) chain_draw_stream_kernel(const ChainParams P) {
  constexpr int kStages = draw_stages<T>();
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t bars[kDrawWarps][kStages];
  using GL = typename Group<T>::L;
  constexpr int LBYTES = kDrawChunk * static_cast<int>(sizeof(T));
  constexpr int STAGE = LBYTES + kDrawChunk * 4;
  constexpr int GPL = kDrawChunk / 4 / 32;  // 4-element groups per lane per chunk
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t NW = gridDim.x * kDrawWarps;
  const uint32_t gw = blockIdx.x * kDrawWarps + warp;
  unsigned char* buf = smem + static_cast<size_t>(warp) * kStages * STAGE;
  uint64_t* bar = bars[warp];
  const int R = P.gamma + 1;
  const uint32_t nchd = P.nchd;

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bar[s], 1);
    mbar_fence_init();
  }
  __syncwarp();
  grid_dependency_wait();  // the decision kernel's list is visible from here
  const uint32_t count = __ldcg(P.ws.draw_count);
  const uint32_t n_items = count * nchd;
  // The list, copied to shared memory when it fits: per-item metadata is then a shared
  // load instead of an L2 round trip in every item's critical path.
  DrawEntry* list_s = reinterpret_cast<DrawEntry*>(smem + static_cast<size_t>(kDrawWarps) * kStages * STAGE);
  const bool cached = count <= static_cast<uint32_t>(kDrawListCache);
  if (cached) {
    for (uint32_t i = threadIdx.x; i < count; i += blockDim.x) {
      list_s[i].loc = __ldcg(&P.ws.draw_list[i].loc);
      list_s[i].row = __ldcg(&P.ws.draw_list[i].row);
    }
  }
  __syncthreads();
  const DrawEntry* list = cached ? list_s : P.ws.draw_list;

  auto issue = [&](uint32_t it, int s, int4 loc) {
    const uint32_t cd = it % nchd;
    const int n = min(kDrawChunk, P.V - static_cast<int>(cd) * kDrawChunk);
    const uint32_t lb = static_cast<uint32_t>(n) * sizeof(T);
    const uint32_t qb = (loc.y < P.gamma) ? static_cast<uint32_t>(n) * 4u : 0u;
    mbar_expect_tx(&bar[s], lb + qb);
    const T* src = static_cast<const T*>(P.logits) + (static_cast<int64_t>(loc.x) * R + loc.y) * P.V +
                   static_cast<int64_t>(cd) * kDrawChunk;
    bulk_copy_g2s(buf + s * STAGE, src, lb, &bar[s]);
    if (qb) {
      const float* qs = P.q + (static_cast<int64_t>(loc.x) * P.gamma + loc.y) * P.V + static_cast<int64_t>(cd) * kDrawChunk;
      bulk_copy_g2s(buf + s * STAGE + LBYTES, qs, qb, &bar[s]);
    }
  };
  uint32_t issued = 0;
  for (uint32_t it = gw; issued < kStages && it < n_items; it += NW, ++issued)
    if (lane == 0) issue(it, static_cast<int>(issued), list[it / nchd].loc);

  uint32_t k = 0;
  for (uint32_t it = gw; it < n_items; it += NW, ++k) {
    const int s = static_cast<int>(k % kStages);
    const uint32_t nx = it + kStages * NW;  // the item this stage is refilled with
    const bool refill = nx < n_items && nx > it;
    int4 nloc = make_int4(0, 0, 0, 0);
    if (lane == 0 && refill) nloc = list[nx / nchd].loc;
    DrawEntry cur;
    cur.loc = list[it / nchd].loc;
    cur.row = list[it / nchd].row;
    if (!mbar_wait(&bar[s], (k / kStages) & 1u)) {
      if (lane == 0) drain_after_timeout(bar, kStages, k, issued, P.ws.error);
      break;
    }
    const uint32_t cd = it % nchd;
    const bool has_q = cur.loc.y < P.gamma;
    const int ng = min(kDrawChunk, P.V - static_cast<int>(cd) * kDrawChunk) / 4;
    const unsigned char* sb = buf + s * STAGE;
    GL lw[GPL];
    float4 qv[GPL];
#pragma unroll
    for (int j = 0; j < GPL; ++j) {
      const int g = lane + 32 * j;
      if (g < ng) {
        lw[j] = reinterpret_cast<const GL*>(sb)[g];
        qv[j] = has_q ? reinterpret_cast<const float4*>(sb + LBYTES)[g] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    __syncwarp();
    if (lane == 0 && refill) {
      fence_proxy_async_smem();
      issue(nx, s, nloc);
    }
    issued += refill ? 1u : 0u;
    float sr = 0.f;
    QCheck qc;
#pragma unroll
    for (int j = 0; j < GPL; ++j) {
      if (lane + 32 * j < ng) {
        float w[4];
        sr += group_weights<T>(lw[j], qv[j], cur.row.x, cur.row.y, cur.row.z, !has_q, w);
        qc.add(qv[j]);
      }
    }
    sr = warp_sum(sr);
    if (__any_sync(0xffffffffu, qc.bad())) {
      sr = kNaN;
      if (lane == 0) atomicOr(P.ws.qbad + cur.loc.x, 1);
    }
    if (lane == 0) P.ws.draw_mass[static_cast<int64_t>(cur.loc.z) * nchd + cd] = sr;
  }
}

// ---------------------------------------------------------------------------------
// finish: one warp per sequence
// ---------------------------------------------------------------------------------

template <typename T>
__global__ void __launch_bounds__(32) chain_finish_kernel(const ChainParams P) {
  grid_launch_dependents();
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x;
  SeqState st;
  st.meta = __ldcg(&P.ws.seq[b].meta);
  st.row = __ldcg(&P.ws.seq[b].row);
  if (st.meta.y != 1) return;
  const int R = P.gamma + 1;
  const int J = st.meta.x;
  const float* dm = P.ws.draw_mass + static_cast<int64_t>(b) * P.nchd;
  int32_t* tok_out = P.out_tokens + static_cast<int64_t>(b) * R;
  const T* lrow = static_cast<const T*>(P.logits) + (static_cast<int64_t>(b) * R + J) * P.V;
  const float* qrow = (J < P.gamma) ? P.q + (static_cast<int64_t>(b) * P.gamma + J) * P.V : nullptr;
  const float invZ = 1.f / st.row.y;
  bool zr = false;
  const int y = draw_from_masses<T, kDrawChunk>(P.V, P.nchd, dm, lrow, qrow, st.row.x, st.row.z, invZ, invZ, st.row.w, lane, zr);
  if (y < 0) {  // a bad draft probability in the drawn row
    if (lane < R) tok_out[lane] = -1;
    if (lane < P.gamma && P.out_p_draft) P.out_p_draft[static_cast<int64_t>(b) * P.gamma + lane] = kNaN;
    if (lane == 0) {
      P.out_J[b] = -1;
      if (P.out_status) P.out_status[b] = st.meta.z | SPECDEC_STATUS_BAD_PROB;
    }
    return;
  }
  if (lane == 0) {
    tok_out[J] = y;
    if (zr && P.out_status) P.out_status[b] = st.meta.z | SPECDEC_STATUS_ZERO_RESIDUAL;
  }
}

// ---------------------------------------------------------------------------------
// Block verification (Art of Guessing, "Block verification", Sun et al.): the same
// statistics pass, then
//   block decide  one CTA per sequence: every row's (m, Z) and argmax, p_k(x_k), the
//                 running weights w_{k+1} = min(1, w_k p_k(x_k) / q_k(x_k)) (w_0 = 1),
//                 every input checked; lists all gamma + 1 rows for the mass pass with
//                 their weights folded into the scale: (w_k p_k - q_k)+ (q_gamma = 0).
//   mass pass     the draw kernel above, over every listed row.
//   block finish  one CTA per sequence: mass_k per row (fp64), survival_k =
//                 mass_k / (mass_k + 1 - w_k) (1 if w_k = 1), n = the longest prefix k
//                 with u[k-1] <= survival_k, and the inverse-CDF draw from row n.
// ---------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kDecideThreads) block_decide_kernel(const ChainParams P) {
  __shared__ float s_m[kStreamMaxRows], s_Z[kStreamMaxRows];
  __shared__ int s_z[kStreamMaxRows];
  grid_launch_dependents();
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = P.gamma + 1;
  const int nch = P.nch;
  const float Tb = P.greedy_only ? 0.f : __ldg(P.temps + b);
  const bool greedy = P.greedy_only || is_greedy(Tb);
  const float c = greedy ? 0.f : kLog2e / Tb;

  // inputs (lane i: position i; lane gamma: the draw's uniform), before the wait
  int x = -1, tok_err = 0, u_err = 0;
  float lx = 0.f, qx = 0.f, ux = 0.f;
  if (warp == 0) {
    if (lane < P.gamma) {
      x = __ldg(P.drafts + static_cast<int64_t>(b) * P.gamma + lane);
      if (x < 0 || x >= P.V) {
        tok_err = SPECDEC_STATUS_BAD_TOKEN;
      } else if (!greedy) {
        lx = Elem<T>::load(static_cast<const T*>(P.logits) + (static_cast<int64_t>(b) * R + lane) * P.V, x);
        qx = __ldg(P.q + (static_cast<int64_t>(b) * P.gamma + lane) * P.V + x);
      }
    }
    if (!greedy && lane < R) {
      ux = __ldg(P.u + static_cast<int64_t>(b) * R + lane);
      if (!(ux >= 0.f && ux < 1.f)) u_err = SPECDEC_STATUS_BAD_UNIFORM;
    }
  }
  grid_dependency_wait();

  for (int r = warp; r < R; r += kDecideThreads / 32) {
    const float4* pp = P.ws.partials + (static_cast<int64_t>(b) * R + r) * nch;
    RowSum acc;
    acc.m = -kInf;
    acc.Z = 0.f;
    acc.z = INT_MAX;
    for (int q = lane; q < nch; q += 32) {
      const float4 f = __ldcg(pp + q);
      RowSum t;
      t.m = f.x;
      t.Z = f.y;
      t.z = __float_as_int(f.z);
      acc = merge(acc, t, c);
    }
    acc = warp_merge(acc, c);
    if (lane == 0) {
      s_m[r] = acc.m;
      s_Z[r] = acc.Z;
      s_z[r] = acc.z;
    }
  }
  __syncthreads();
  if (warp != 0) return;

  float m = -kInf, Z = 0.f;
  int z = INT_MAX, row_err = 0;
  if (lane < R) {
    m = s_m[lane];
    Z = s_Z[lane];
    z = s_z[lane];
    if (!(m == m) || m == kInf) row_err = SPECDEC_STATUS_BAD_LOGIT;
    else if (m == -kInf) row_err = SPECDEC_STATUS_EMPTY_ROW;
  }
  // every row, draft and uniform is read by the rule: every error is reported
  int err = __reduce_or_sync(0xffffffffu, row_err | tok_err | u_err);
  const bool bad_T = !P.greedy_only && !(Tb - Tb == 0.f);
  if (bad_T) err = SPECDEC_STATUS_BAD_TEMPERATURE;
  int32_t* tok_out = P.out_tokens + static_cast<int64_t>(b) * R;
  float* pd_out = P.out_p_draft ? P.out_p_draft + static_cast<int64_t>(b) * P.gamma : nullptr;

  if (greedy || bad_T) {
    // greedy matching (a one-hot target reduces the block rule to it)
    const bool miss = lane < P.gamma && x != z;
    const unsigned mm = __ballot_sync(0xffffffffu, miss);
    const int J = err ? -1 : (mm ? __ffs(mm) - 1 : P.gamma);
    const int zJ = __shfl_sync(0xffffffffu, z, J < 0 ? 0 : J);
    if (lane < R) tok_out[lane] = (J < 0) ? -1 : (lane < J ? x : (lane == J ? zJ : -1));
    if (lane < P.gamma && pd_out) pd_out[lane] = kNaN;
    if (lane == 0) {
      P.out_J[b] = J;
      if (P.out_status) P.out_status[b] = err;
      SeqState sq;
      sq.meta = make_int4(J, 0, err, 0);
      sq.row = make_float4(0.f, 0.f, 0.f, 0.f);
      P.ws.seq[b] = sq;
    }
    return;
  }

  // p_k(x_k), the ratios and the running weights (one serial pass over the positions)
  float px = kNaN;
  int warn = 0;
  float ratio = 0.f;
  if (lane < P.gamma && !tok_err) {
    px = ex2((lx - m) * c) / Z;
    if (qx == 0.f) {
      warn = SPECDEC_STATUS_ZERO_Q;
      ratio = px > 0.f ? kInf : 0.f;
    } else {
      ratio = px / qx;
    }
  }
  warn = __reduce_or_sync(0xffffffffu, warn);
  float w = 1.f, wk = 1.f;  // wk: this lane's w_lane
  for (int k = 0; k < P.gamma; ++k) {
    const float rk = __shfl_sync(0xffffffffu, ratio, k);
    w = (w == 0.f) ? 0.f : fminf(1.f, w * rk);
    if (lane == k + 1) wk = w;
  }
  if (lane < P.gamma && pd_out) pd_out[lane] = err ? kNaN : px;
  if (lane < R) P.ws.block_rows[static_cast<int64_t>(b) * R + lane] = make_float4(m, Z, wk, 0.f);
  // Rows for the mass pass: the gamma rows with q always (their q rows are checked even
  // when the sequence already failed), the bonus row only for a clean sequence.
  const int nent = err ? P.gamma : R;
  unsigned base = 0;
  if (lane == 0) base = atomicAdd(P.ws.draw_count, static_cast<unsigned>(nent));
  base = __shfl_sync(0xffffffffu, base, 0);
  if (lane < nent) {
    DrawEntry d;
    d.loc = make_int4(b, lane, b * R + lane, 0);
    d.row = make_float4(m, c, wk / Z, 0.f);
    P.ws.draw_list[base + lane] = d;
  }
  if (lane == 0) {
    SeqState sq;
    sq.meta = make_int4(-1, 2, err | warn, 0);
    sq.row = make_float4(0.f, 0.f, c, 0.f);
    P.ws.seq[b] = sq;
  }
}

template <typename T>
__global__ void __launch_bounds__(kDecideThreads) block_finish_kernel(const ChainParams P) {
  __shared__ double s_mass[kStreamMaxRows];
  grid_launch_dependents();
  grid_dependency_wait();
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  SeqState st;
  st.meta = __ldcg(&P.ws.seq[b].meta);
  st.row = __ldcg(&P.ws.seq[b].row);
  if (st.meta.y != 2) return;
  const int R = P.gamma + 1;
  const int nchd = P.nchd;
  int status = st.meta.z;
  if (__ldcg(P.ws.qbad + b)) status |= SPECDEC_STATUS_BAD_PROB;
  int32_t* tok_out = P.out_tokens + static_cast<int64_t>(b) * R;
  if (status & SPECDEC_STATUS_ERROR_MASK) {  // errors only: warnings describe a clean round
    status &= SPECDEC_STATUS_ERROR_MASK;
    if (warp == 0) {
      if (lane < R) tok_out[lane] = -1;
      if (lane < P.gamma && P.out_p_draft) P.out_p_draft[static_cast<int64_t>(b) * P.gamma + lane] = kNaN;
      if (lane == 0) {
        P.out_J[b] = -1;
        if (P.out_status) P.out_status[b] = status;
      }
    }
    return;
  }
  // mass_k of every row (fp64, fixed order: lane-contiguous runs, then the warp)
  for (int k = warp; k < R; k += kDecideThreads / 32) {
    const float* dm = P.ws.draw_mass + (static_cast<int64_t>(b) * R + k) * nchd;
    const int cpl = (nchd + 31) / 32;
    const int q0 = min(lane * cpl, nchd), q1 = min(q0 + cpl, nchd);
    double mine = 0.0;
    for (int q = q0; q < q1; ++q) mine += static_cast<double>(__ldcg(dm + q));
    const double tot = warp_incl_scan(mine, lane);
    if (lane == 31) s_mass[k] = tot;
  }
  __syncthreads();
  if (warp != 0) return;
  // survival of every prefix and the longest surviving one
  float4 br = make_float4(0.f, 1.f, 1.f, 0.f);
  if (lane < R) br = __ldcg(P.ws.block_rows + static_cast<int64_t>(b) * R + lane);
  const double wk = static_cast<double>(br.z);
  bool survived = false;
  if (lane >= 1 && lane < R) {
    const double mass = s_mass[lane];
    const double surv = (wk < 1.0) ? mass / (mass + 1.0 - wk) : 1.0;
    const float uk = __ldg(P.u + static_cast<int64_t>(b) * R + lane - 1);
    survived = static_cast<double>(uk) <= surv;
  }
  const unsigned sv = __ballot_sync(0xffffffffu, survived);
  const int n = sv ? 31 - __clz(sv) : 0;
  const float mN = __shfl_sync(0xffffffffu, br.x, n), zN = __shfl_sync(0xffffffffu, br.y, n);
  const float wN = __shfl_sync(0xffffffffu, br.z, n);
  const float c = st.row.z;
  const T* lrow = static_cast<const T*>(P.logits) + (static_cast<int64_t>(b) * R + n) * P.V;
  const float* qrow = (n < P.gamma) ? P.q + (static_cast<int64_t>(b) * P.gamma + n) * P.V : nullptr;
  const float uG = __ldg(P.u + static_cast<int64_t>(b) * R + P.gamma);
  bool zr = false;
  const int y = draw_from_masses<T, kDrawChunk>(P.V, nchd, P.ws.draw_mass + (static_cast<int64_t>(b) * R + n) * nchd, lrow, qrow, mN,
                                    c, wN / zN, 1.f / zN, uG, lane, zr);
  const int x = (lane < P.gamma) ? __ldg(P.drafts + static_cast<int64_t>(b) * P.gamma + lane) : -1;
  if (lane < R) tok_out[lane] = lane < n ? x : (lane == n ? y : -1);
  if (lane == 0) {
    P.out_J[b] = n;
    if (P.out_status) P.out_status[b] = status | (zr ? SPECDEC_STATUS_ZERO_RESIDUAL : 0);
  }
}

// Raise a kernel's dynamic shared-memory limit once per device; `configured` must be a
// flag set private to that kernel.
cudaError_t set_smem(const void* kernel, int bytes, unsigned long long& configured) {
  int dev = 0;
  cudaGetDevice(&dev);
  const unsigned long long bit = 1ull << (dev & 63);
  if (configured & bit) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) configured |= bit;
  return e;
}

template <typename T>
cudaError_t launch_stats_t(const ChainParams& P, cudaStream_t stream) {
  constexpr int smem = kStatsWarps * kStatsStages * kStatsChunkBytes;
  static unsigned long long configured = 0;
  cudaError_t e = set_smem(reinterpret_cast<const void*>(chain_stats_stream_kernel<T>), smem, configured);
  if (e != cudaSuccess) return e;
  return launch_kernel(chain_stats_stream_kernel<T>, dim3(P.grid_stats), dim3(kStatsWarps * 32), smem,
                       stream, 0, P);
}

template <typename T>
cudaError_t launch_draw_t(const ChainParams& P, cudaStream_t stream) {
  constexpr int smem = draw_smem_bytes<T>();
  static unsigned long long configured = 0;
  cudaError_t e = set_smem(reinterpret_cast<const void*>(chain_draw_stream_kernel<T>), smem, configured);
  if (e != cudaSuccess) return e;
  return launch_kernel(chain_draw_stream_kernel<T>, dim3(P.grid_draw), dim3(kDrawWarps * 32), smem, stream, 1, P);
}

}  // namespace

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

cudaError_t launch_chain_stream_stats(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream) {
  return ldt == SPECDEC_BF16 ? launch_stats_t<uint16_t>(P, stream) : launch_stats_t<float>(P, stream);
}

cudaError_t launch_chain_stream_decide(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream) {
  if (ldt == SPECDEC_BF16)
    return launch_kernel(chain_decide_kernel<uint16_t>, dim3(P.B), dim3(kDecideThreads), 0, stream, 1, P);
  return launch_kernel(chain_decide_kernel<float>, dim3(P.B), dim3(kDecideThreads), 0, stream, 1, P);
}

cudaError_t launch_chain_stream_draw(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream) {
  return ldt == SPECDEC_BF16 ? launch_draw_t<uint16_t>(P, stream) : launch_draw_t<float>(P, stream);
}

cudaError_t launch_block_decide(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream) {
  if (ldt == SPECDEC_BF16)
    return launch_kernel(block_decide_kernel<uint16_t>, dim3(P.B), dim3(kDecideThreads), 0, stream, 1, P);
  return launch_kernel(block_decide_kernel<float>, dim3(P.B), dim3(kDecideThreads), 0, stream, 1, P);
}

cudaError_t launch_block_finish(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream) {
  if (ldt == SPECDEC_BF16)
    return launch_kernel(block_finish_kernel<uint16_t>, dim3(P.B), dim3(kDecideThreads), 0, stream, 1, P);
  return launch_kernel(block_finish_kernel<float>, dim3(P.B), dim3(kDecideThreads), 0, stream, 1, P);
}

cudaError_t launch_chain_stream_finish(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream) {
  if (ldt == SPECDEC_BF16)
    return launch_kernel(chain_finish_kernel<uint16_t>, dim3(P.B), dim3(32), 0, stream, 1, P);
  return launch_kernel(chain_finish_kernel<float>, dim3(P.B), dim3(32), 0, stream, 1, P);
}

}  // namespace specdec
