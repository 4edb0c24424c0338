// Chain verification that reads only the rows a round needs.
//
// SD 20.5, "A whole round of speculative sampling": the one-token rule is applied to the
// drafts left to right and the round stops at the first rejection; the drafts after it
// are discarded, so their target rows are never needed.  This kernel follows that order
// literally, as a dataflow of TASKS:
//
//   row task (b, i)   the softmax statistics of row i of sequence b and the test of draft
//                     i: accept iff u_i * q_i(x_i) < p_i(x_i) (greedy: x_i == argmax).  An
//                     acceptance makes row i + 1 the next task; a rejection, or row gamma,
//                     queues the draw task (b, i) (a greedy sequence emits the argmax).
//   draw task (b, J)  the residual weights (p_J - q_J)+ (q == 0 for the bonus row; SD 20.5,
//                     "The speculative sampling rule") and the inverse-CDF draw: the
//                     smallest k with C_k > u * S.
//
// A task is run by a TEAM: one group of warps in each of the kSeqCluster CTAs of a
// thread-block cluster (one CTA per SM).  Member r owns the r-th contiguous part of the
// row.  Each warp streams its chunks through a bulk-copy pipeline (cp.async.bulk copies
// in flight on mbarriers); each lane keeps a running maximum and sum of
// 2^((l - m) * log2(e) / T) (or the lowest index of the maximum), or, for a draw, sums
// residual weights per 512-element chunk.  Members exchange their 16-byte summaries by
// st.async into each other's shared memory (distributed shared memory); every member
// merges them in member order, so all hold the same bits and take the same decision.
// The member whose part holds u * S finds the drawn token.
//
// A team follows its sequence's chain row after row.  When the chain ends, the team
// takes new work from two ticket queues: sequence starts first, then queued draws.  So
// every chain starts early, and the draws fill the machine behind the chains.
//
// The logits and draft probabilities may also sit in pinned host memory (kHost): the
// kernel then reads them over the host link itself, only the rows the round needs, with
// per-lane 16-byte cp.async copies into the same stages (bulk copies are kept to device
// memory) and plain loads for single elements.

#include <climits>

#include "specdec_device.cuh"
#include "specdec_internal.h"

namespace specdec {

namespace {

constexpr uint32_t kNegInfBf16x2 = 0xFF80FF80u;
constexpr float kNaN = __builtin_nanf("");
constexpr int kWarpsPerGroup = kSeqWarps / kSeqGroups;
constexpr int kGroupThreads = kWarpsPerGroup * 32;
constexpr int kC = kSeqCluster;
// Copies a warp keeps in flight for a draw task (a row task keeps kSeqStages).  While both
// stream, the rows -- the chains, which are the critical path -- get the larger share of
// the bandwidth; the draws fill in behind them.  A draw taken while other teams wait for
// work (the machine has bandwidth to spare) keeps kSeqStages too.
constexpr int kSeqDrawStages = 2;
static_assert(kSeqDrawStages >= 1 && kSeqDrawStages <= kSeqStages, "draw copies use the row stages");
static_assert(kSeqWarps % kSeqGroups == 0, "groups must split the warps evenly");
static_assert(kC >= 1 && kC <= 8, "portable cluster sizes only");

__device__ __forceinline__ bool is_greedy(float T) { return !(T >= SPECDEC_GREEDY_TEMPERATURE); }

// Loads of the logits and q rows: through the read-only path from device memory, plain
// global loads (cached in L2 only) when the rows may sit in host memory.
template <bool kHost, typename X>
__device__ __forceinline__ X load_in(const X* p) {
  if constexpr (kHost) return __ldcg(p);
  else return __ldg(p);
}
template <bool kHost, typename T>
__device__ __forceinline__ float load_elem(const T* row, int64_t k) {
  if constexpr (sizeof(T) == 2) return __uint_as_float(static_cast<uint32_t>(load_in<kHost>(row + k)) << 16);
  else return load_in<kHost>(row + k);
}

// One 16-byte asynchronous copy of global (or mapped host) memory into shared memory, and
// the arrival of this thread on an mbarrier once all its earlier such copies have landed
// (the barrier counts one arrival per copying thread).
__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Barrier over the threads of one group (named barriers 1.., 0 stays __syncthreads).
__device__ __forceinline__ void group_sync(int group) {
  asm volatile("bar.sync %0, %1;" ::"r"(group + 1), "r"(kGroupThreads) : "memory");
}
// Barrier over the group that also returns whether any of its threads passed `v`.
__device__ __forceinline__ bool group_any(int group, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(group + 1), "r"(kGroupThreads)
      : "memory");
  return r != 0;
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
__device__ __forceinline__ float warp_incl_scan(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// (max, normaliser, lowest argmax) of a part of a row, and the merge of two parts.
// Every exponent on this path is l * c - rnd(m * c), one fused multiply-add against the
// rounded product of the maximum in force; a rescale between two maxima multiplies by
// 2^(rnd(m_old * c) - rnd(m_new * c)).  The rounding of m * c then shifts every term of
// a row alike, and cancels in p = 2^(l_x * c - rnd(m * c)) / Z.
struct RowSum {
  float m, Z;
  int z;
};
__device__ __forceinline__ RowSum merge(const RowSum& a, const RowSum& b, float c) {
  RowSum r;
  r.m = max_nan(a.m, b.m);
  const float mc = __fmul_rn(r.m, c);
  const float za = (a.m > -kInf) ? a.Z * ex2(__fsub_rn(__fmul_rn(a.m, c), mc)) : 0.f;
  const float zb = (b.m > -kInf) ? b.Z * ex2(__fsub_rn(__fmul_rn(b.m, c), mc)) : 0.f;
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
// index order; the chunk masses and the final scan both use it.  nmc = -rnd(m_J * c);
// with q == 0 (the bonus row, or a zero residual) the weights are p itself.
template <typename T>
__device__ __forceinline__ float group_weights(const typename Group<T>::L& lw, const float4& q4, float nmc,
                                               float c, float invZ, bool no_q, float (&w)[4]) {
  float l[4];
  Group<T>::unpack(lw, l);
  const unsigned long long c2 = f2pack(c, c), nmc2 = f2pack(nmc, nmc), niz2 = f2pack(-invZ, -invZ);
  const unsigned long long q01 = no_q ? 0ull : f2pack(q4.x, q4.y), q23 = no_q ? 0ull : f2pack(q4.z, q4.w);
  float acc = 0.f;
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    float y0, y1;
    f2unpack(f2fma(f2pack(l[2 * p], l[2 * p + 1]), c2, nmc2), y0, y1);
    float r0, r1;  // q - p
    f2unpack(f2fma(f2pack(ex2(y0), ex2(y1)), niz2, p == 0 ? q01 : q23), r0, r1);
    w[2 * p] = fmaxf(-r0, 0.f);
    w[2 * p + 1] = fmaxf(-r1, 0.f);
    acc += w[2 * p];
    acc += w[2 * p + 1];
  }
  return acc;
}

// Shared state of one group (one team member).  Its layout is the same in every CTA, so
// a member's slot in another CTA is this one's address mapped to that CTA.
struct GroupShared {
  float4 slot[2][kC];           // summary exchange slots by parity, one per member
  uint64_t xbar[2];             // their mbarriers
  float4 mbox[2][2];            // the next task's 32-byte entry, by task parity
  uint64_t mbar_box[2];         // their mbarriers
  RowSum wsum[kWarpsPerGroup];  // per-warp row summaries
  // per task parity: draft token bits, its logit, its q, u_i, u_gamma, input error bits
  float gq[2][8];
  float mass[2][kSeqMaxDrawChunks];  // draw: mass per chunk of this member's part, by task parity
};

// This group's side of a team: its member index and the exchange sequence number.
struct Team {
  uint32_t rank = 0;
  uint32_t xk = 0;
  bool ok = true;  // false once a bounded wait gave up
};

// Every member contributes 16 bytes (`mine`, taken from the first thread of the group);
// on return every thread of the group can read all contributions in gs.slot[par][*].
// Two parities alternate and a group barrier closes each exchange; a member sends into a
// parity only after every member finished the exchange before it, so a slot is never
// rewritten while a thread may still read it.
__device__ int exchange(GroupShared& gs, Team& tm, const float4& mine, int group, int gwarp, int lane,
                        unsigned* error) {
  const int par = static_cast<int>(tm.xk & 1u);
  const uint32_t phase = (tm.xk >> 1) & 1u;
  ++tm.xk;
  bool waited = true;
  if (tm.ok) {
    if (gwarp == 0 && lane == 0) {
      mbar_expect_tx(&gs.xbar[par], kC * 16);
      const uint32_t sa = smem_addr(&gs.slot[par][tm.rank]);
      const uint32_t ba = smem_addr(&gs.xbar[par]);
#pragma unroll
      for (int r = 0; r < kC; ++r) st_async_16(cluster_map(sa, r), mine, cluster_map(ba, r));
    }
    waited = mbar_wait_cluster(&gs.xbar[par], phase);
  }
  if (group_any(group, !waited)) {
    if (gwarp == 0 && lane == 0) atomicOr(error, 2u);
    tm.ok = false;
  }
  return par;
}

// One warp's bulk-copy pipeline: kSeqStages stages of kSeqChunkBytes in shared memory.
// `k` counts completed stages and `issued` issued ones, over the kernel's lifetime.
struct Pipe {
  unsigned char* buf;
  uint64_t* bar;
  uint32_t k = 0, issued = 0;
  bool ok = true;  // false once a bounded wait gave up

  __device__ __forceinline__ unsigned char* stage(uint32_t i) { return buf + (i % kSeqStages) * kSeqChunkBytes; }
  __device__ __forceinline__ uint64_t* sbar(uint32_t i) { return bar + (i % kSeqStages); }
  __device__ __forceinline__ uint32_t in_flight() const { return issued - k; }
  // Issue one copy group (one or two copies) into the next stage: bulk copies by one lane,
  // or (kHost) 16-byte copies by every lane, each of which then arrives on the stage's
  // barrier.  The fence orders this warp's earlier reads of that stage (completed by a
  // __syncwarp) before the copy.
  template <bool kHost>
  __device__ __forceinline__ void issue(const void* a, uint32_t na, const void* b, uint32_t nb, int off_b, int lane) {
    uint64_t* br = sbar(issued);
    unsigned char* dst = stage(issued);
    if constexpr (kHost) {
      const char* ca = static_cast<const char*>(a);
      const char* cb = static_cast<const char*>(b);
      for (uint32_t o = 16u * lane; o < na; o += 512u) cp_async_16(dst + o, ca + o);
      for (uint32_t o = 16u * lane; o < nb; o += 512u) cp_async_16(dst + off_b + o, cb + o);
      cp_async_arrive(br);
    } else if (lane == 0) {
      fence_proxy_async_smem();
      mbar_expect_tx(br, na + nb);
      bulk_copy_g2s(dst, a, na, br);
      if (nb) bulk_copy_g2s(dst + off_b, b, nb, br);
    }
  }
  __device__ __forceinline__ bool wait() { return mbar_wait(sbar(k), (k / kSeqStages) & 1u); }
};

enum : int { kTaskRow = 1, kTaskDraw = 2, kTaskDrawP = 3 };

// A task entry: 32 bytes, in the global rings and in a team's mailbox.
//   e0 = (sequence b (-1: no more work), row | kind << 8 | warnings << 16, m, Z)
//   e1 = (T, 0, 0, 0)
// (m, Z) are the drawn row's maximum and normaliser for draw tasks; the warnings are
// the sequence's status bits above the error byte, shifted down by 8.
struct Entry {
  int b, row, kind, warn;
  float m, Z, T;
  int deep = 0;  // a draw taken while teams wait for work: all kSeqStages copies in flight
};
__device__ __forceinline__ void pack_entry(const Entry& e, float4& e0, float4& e1) {
  e0 = make_float4(__int_as_float(e.b), __int_as_float(e.row | (e.kind << 8) | (e.warn << 16)), e.m, e.Z);
  e1 = make_float4(e.T, 0.f, 0.f, 0.f);
}
__device__ __forceinline__ Entry unpack_entry(const float4& e0, const float4& e1) {
  Entry e;
  e.b = __float_as_int(e0.x);
  const int bits = __float_as_int(e0.y);
  e.row = bits & 0xff;
  e.kind = (bits >> 8) & 0xff;
  e.warn = bits >> 16;
  e.m = e0.z;
  e.Z = e0.w;
  e.T = e1.x;
  e.deep = __float_as_int(e1.y);
  return e;
}

__device__ __forceinline__ unsigned ld_relaxed(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Work that any team may take: the start of a sequence (its row 0; ticket s < B is
// sequence s) and published draw tasks (draw ticket d is the d-th published draw).
// Tickets are handed out by atomicAdd, so claiming never retries.  A team takes a ticket
// only when it has no task; a draw ticket taken before its draw is published is waited
// for then, and that draw comes from a team still following its chain, so no team ever
// waits on work that it must produce itself.
struct Queue {
  unsigned *start_ticket, *pub_draws, *draw_ticket, *finished;
  int* ready_draws;
  float4* ring_draws;
  int B;
};
constexpr int kDrawTag = 1 << 30;

__device__ __forceinline__ int take_ticket(const Queue& q) {
  if (ld_relaxed(q.start_ticket) < static_cast<unsigned>(q.B)) {
    const unsigned s = atomicAdd(q.start_ticket, 1u);
    if (s < static_cast<unsigned>(q.B)) return static_cast<int>(s);
  }
  return kDrawTag | static_cast<int>(atomicAdd(q.draw_ticket, 1u));
}

// The entry behind a ticket, waiting until it is published: 1 = ready, -1 = every
// sequence has finished (no more work), -2 = the bounded wait gave up.
__device__ int resolve_ticket(const ChainParams& P, const Queue& q, int tk, float4& e0, float4& e1) {
  if (!(tk & kDrawTag)) {
    Entry e;
    e.b = tk;
    e.row = 0;
    e.kind = kTaskRow;
    e.warn = 0;
    e.m = 0.f;
    e.Z = 1.f;
    e.T = P.greedy_only ? 0.f : __ldg(P.temps + tk);
    pack_entry(e, e0, e1);
    return 1;
  }
  const int d = tk & ~kDrawTag;
  uint64_t t0 = 0;
  for (;;) {
    if (d < 2 * q.B && ld_acquire(q.ready_draws + d) != 0) {
      const float4* ent = q.ring_draws + 2 * static_cast<int64_t>(d);
      e0 = __ldcg(ent);
      e1 = __ldcg(ent + 1);
      // teams waiting for work: the machine has bandwidth to spare, stream the draw deep
      const int idle = static_cast<int>(ld_relaxed(q.draw_ticket) - ld_relaxed(q.pub_draws));
      e1.y = __int_as_float(idle > 0 ? 1 : 0);
      return 1;
    }
    if (ld_relaxed(q.finished) >= static_cast<unsigned>(q.B)) return -1;
    if (t0 == 0) t0 = global_timer_ns();
    else if (global_timer_ns() - t0 > kMaxWaitNs) return -2;
    __nanosleep(128);
  }
}

__device__ void publish_draw(const Queue& q, const Entry& e) {
  float4 e0, e1;
  pack_entry(e, e0, e1);
  const unsigned k = atomicAdd(q.pub_draws, 1u);
  float4* ent = q.ring_draws + 2 * static_cast<int64_t>(k);
  __stcg(ent, e0);
  __stcg(ent + 1, e1);
  st_release(q.ready_draws + k, 1);
}

// The team leader hands a task entry to every member's mailbox of the given parity.
__device__ __forceinline__ void send_entry(GroupShared& gs, int par, const float4& e0, const float4& e1) {
  const uint32_t sa = smem_addr(&gs.mbox[par][0]);
  const uint32_t ba = smem_addr(&gs.mbar_box[par]);
#pragma unroll
  for (int r = 0; r < kC; ++r) {
    st_async_16(cluster_map(sa, r), e0, cluster_map(ba, r));
    st_async_16(cluster_map(sa + 16, r), e1, cluster_map(ba, r));
  }
}

// This member's copies of one task: the logits row (or drawn row) and, for a residual
// draw, the q row; the member's chunk range [lo, hi) (4 KB chunks for a row, 512-element
// chunks for a draw); this warp's jobs are the chunks lo + gwarp, lo + gwarp + W, ...
struct Task {
  int kind = 0;
  const char* src = nullptr;
  const float* q = nullptr;
  int lo = 0, hi = 0, n = 0;
};

template <typename T, bool kHost>
__device__ __forceinline__ void issue_job(Pipe& pp, const Task& t, int j, int gwarp, int lane, int V,
                                          int64_t row_bytes) {
  constexpr int LB = kSeqDrawChunk * static_cast<int>(sizeof(T));
  if (kHost || lane == 0) {
    const int ch = t.lo + gwarp + j * kWarpsPerGroup;
    if (t.kind == kTaskRow) {
      const uint32_t nb = static_cast<uint32_t>(
          min(static_cast<int64_t>(kSeqChunkBytes), row_bytes - static_cast<int64_t>(ch) * kSeqChunkBytes));
      pp.issue<kHost>(t.src + static_cast<int64_t>(ch) * kSeqChunkBytes, nb, nullptr, 0, 0, lane);
    } else {
      const int n = min(kSeqDrawChunk, V - ch * kSeqDrawChunk);
      const int64_t off = static_cast<int64_t>(ch) * kSeqDrawChunk;
      pp.issue<kHost>(t.src + off * static_cast<int64_t>(sizeof(T)), static_cast<uint32_t>(n) * sizeof(T),
                      t.q ? t.q + off : nullptr, t.q ? static_cast<uint32_t>(n) * 4u : 0u, LB, lane);
    }
  }
  ++pp.issued;
}

// One 4 KB chunk of a row into this lane's running (max, sum, argmax).
template <typename T>
__device__ __forceinline__ void row_chunk(const uint4 (&w)[kSeqChunkBytes / 512], int nv, int ch, bool greedy,
                                          float c, int lane, float& ml, float& Zl, int& zl) {
  constexpr int VEC = Vec<T>::n;
  constexpr int VPL = kSeqChunkBytes / 16 / 32;
  constexpr int EPC = kSeqChunkBytes / static_cast<int>(sizeof(T));
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
      const float mcn = __fmul_rn(mn, c);
      if (mn != ml) Zl = (ml > -kInf) ? Zl * ex2(__fsub_rn(__fmul_rn(ml, c), mcn)) : 0.f;
      ml = mn;
      const unsigned long long nmc2 = f2pack(-mcn, -mcn), c2 = f2pack(c, c);
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
          f2unpack(f2fma(x2, c2, nmc2), y0, y1);
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

// fp32 scan of this member's chunk masses (first warp): each lane sums a contiguous run
// of chunks.  The search repeats exactly this arithmetic, so the member's total and the
// search's running prefixes agree to the bit.
struct LocalScan {
  int c0, c1;
  float mine, incl, total;
};
__device__ __forceinline__ LocalScan local_scan(const float* mass, int n, int lane) {
  LocalScan s;
  const int cpl = (n + 31) / 32;
  s.c0 = min(lane * cpl, n);
  s.c1 = min(s.c0 + cpl, n);
  s.mine = 0.f;
  for (int q = s.c0; q < s.c1; ++q) s.mine += mass[q];
  s.incl = warp_incl_scan(s.mine, lane);
  s.total = __shfl_sync(0xffffffffu, s.incl, 31);
  return s;
}

// Inverse-CDF search inside this member's part (first warp of the chosen member): the
// chunk whose running mass (from `base`, the mass of all earlier members) first exceeds
// `target`, then the element inside it.  If rounding leaves no such element, the last
// positive-weight element of the part is taken.
template <typename T, bool kHost>
__device__ int local_search(const T* lrow, const float* qrow, int V, int d0, int n, float base, float target,
                            float mJ, float c, float invZ, bool no_q, const float* mass, int lane) {
  using GL = typename Group<T>::L;
  constexpr int GPL = kSeqDrawChunk / 4 / 32;
  const LocalScan s = local_scan(mass, n, lane);
  int cstar = -1, lastpos = -1;
  float cbase = 0.f, prelast = 0.f, pre = base + (s.incl - s.mine);
  for (int q = s.c0; q < s.c1; ++q) {
    const float w = mass[q];
    if (w > 0.f) { lastpos = q; prelast = pre; }
    if (cstar < 0 && pre + w > target) { cstar = q; cbase = pre; }
    pre += w;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, cstar >= 0);
  if (hit) {
    const int fl = __ffs(hit) - 1;
    cstar = __shfl_sync(0xffffffffu, cstar, fl);
    cbase = __shfl_sync(0xffffffffu, cbase, fl);
  } else {  // rounding put u * S at or past the end of the part: last chunk with mass
    const int best = warp_max_int(lastpos);
    const unsigned owner = __ballot_sync(0xffffffffu, lastpos == best && best >= 0);
    cstar = best < 0 ? 0 : best;
    cbase = owner ? __shfl_sync(0xffffffffu, prelast, __ffs(owner) - 1) : base;
  }
  const int k0 = (d0 + cstar) * kSeqDrawChunk;
  const int ng = min(kSeqDrawChunk, V - k0) / 4;
  float w[GPL][4], gsum[GPL];
  float lane_tot = 0.f;
#pragma unroll
  for (int j = 0; j < GPL; ++j) {
    const int g = lane * GPL + j;
    gsum[j] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) w[j][e] = 0.f;
    if (g < ng) {
      const GL lw = load_in<kHost>(reinterpret_cast<const GL*>(lrow + k0) + g);
      const float4 q4 = no_q ? make_float4(0.f, 0.f, 0.f, 0.f) : load_in<kHost>(reinterpret_cast<const float4*>(qrow + k0) + g);
      gsum[j] = group_weights<T>(lw, q4, -__fmul_rn(mJ, c), c, invZ, no_q, w[j]);
      lane_tot += gsum[j];
    }
  }
  int last_pos = -1;
#pragma unroll
  for (int j = 0; j < GPL; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (w[j][e] > 0.f) last_pos = k0 + 4 * (lane * GPL + j) + e;
  const float gincl = warp_incl_scan(lane_tot, lane);
  const unsigned ghit = __ballot_sync(0xffffffffu, cbase + gincl > target);
  int y = -1;
  if (ghit) {
    const int fl = __ffs(ghit) - 1;
    if (lane == fl) {
      float p2 = cbase + (gincl - lane_tot);
#pragma unroll
      for (int j = 0; j < GPL; ++j) {
        if (y < 0 && p2 + gsum[j] > target) {
          float run = 0.f;
          int lastp = -1;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            run += w[j][e];
            if (w[j][e] > 0.f) lastp = k0 + 4 * (lane * GPL + j) + e;
            if (y < 0 && p2 + run > target) y = k0 + 4 * (lane * GPL + j) + e;
          }
          if (y < 0) y = lastp;
        }
        p2 += gsum[j];
      }
    }
    y = __shfl_sync(0xffffffffu, y, fl);
  }
  if (y < 0) y = warp_max_int(last_pos);
  return y;
}

// A member's draw total (fp32), a flag and the leader's unclaimed sequence as one 16-byte
// exchange payload.
__device__ __forceinline__ float4 pack_total(float t, int flag, int bn) {
  return make_float4(t, 0.f, __int_as_float(flag), __int_as_float(bn));
}
__device__ __forceinline__ float unpack_total(const float4& v) { return v.x; }

// ---------------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------------
template <typename T, bool kHost>
__global__ void __launch_bounds__(kSeqWarps * 32, 1) chain_seq_kernel(const ChainParams P) {
  using GL = typename Group<T>::L;
  constexpr int VPL = kSeqChunkBytes / 16 / 32;
  constexpr int GPL = kSeqDrawChunk / 4 / 32;
  constexpr int LB = kSeqDrawChunk * static_cast<int>(sizeof(T));
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t bars[kSeqWarps][kSeqStages];
  __shared__ GroupShared gshared[kSeqGroups];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int group = warp / kWarpsPerGroup, gwarp = warp % kWarpsPerGroup;
  GroupShared& gs = gshared[group];
  Pipe pp;
  pp.buf = smem + static_cast<size_t>(warp) * kSeqStages * kSeqChunkBytes;
  pp.bar = bars[warp];
  // Launched without the cluster shape this code maps addresses for: touch nothing.
  if (cluster_size() != static_cast<uint32_t>(kC)) {
    if (threadIdx.x == 0) atomicOr(P.ws.error, 4u);
    return;
  }
  Team tm;
  tm.rank = cluster_rank();
  const bool first = gwarp == 0 && lane == 0;  // this member's first thread
  const bool leader = tm.rank == 0 && first;   // the team's first thread
  if (lane == 0) {
    for (int s = 0; s < kSeqStages; ++s) mbar_init(&pp.bar[s], kHost ? 32 : 1);
    if (gwarp == 0) {
      mbar_init(&gs.xbar[0], 1);
      mbar_init(&gs.xbar[1], 1);
      mbar_init(&gs.mbar_box[0], 1);
      mbar_init(&gs.mbar_box[1], 1);
    }
    mbar_fence_init();
  }
  // Every member's barriers exist before any member writes into another's shared memory.
  cluster_sync_all();

  const int R = P.gamma + 1;
  const int V = P.V;
  const int64_t row_bytes = static_cast<int64_t>(V) * sizeof(T);
  const int nch = static_cast<int>((row_bytes + kSeqChunkBytes - 1) / kSeqChunkBytes);
  const int nchd = (V + kSeqDrawChunk - 1) / kSeqDrawChunk;
  const int c0 = static_cast<int>(static_cast<int64_t>(nch) * tm.rank / kC);
  const int c1 = static_cast<int>(static_cast<int64_t>(nch) * (tm.rank + 1) / kC);
  const int d0 = static_cast<int>(static_cast<int64_t>(nchd) * tm.rank / kC);
  const int d1 = static_cast<int>(static_cast<int64_t>(nchd) * (tm.rank + 1) / kC);
  const char* logits = static_cast<const char*>(P.logits);
  Queue qu;
  qu.start_ticket = P.ws.queue;
  qu.pub_draws = P.ws.queue + 1;
  qu.draw_ticket = P.ws.queue + 2;
  qu.finished = P.ws.queue + 3;
  qu.ready_draws = P.ws.ready;
  qu.ring_draws = P.ws.ring;
  qu.B = P.B;

  // drafts to verify for sequence b: gamma, or its own count (the bonus row is row gb)
  auto gamma_of = [&](int b) { return P.gammas ? __ldg(P.gammas + b) : P.gamma; };
  auto make_task = [&](const Entry& e) {
    Task t;
    t.kind = e.kind;
    t.src = logits + (static_cast<int64_t>(e.b) * R + e.row) * row_bytes;
    t.q = (e.kind == kTaskDraw && e.row < gamma_of(e.b)) ? P.q + (static_cast<int64_t>(e.b) * P.gamma + e.row) * V
                                                          : nullptr;
    t.lo = (e.kind == kTaskRow) ? c0 : d0;
    t.hi = (e.kind == kTaskRow) ? c1 : d1;
    t.n = (t.hi > t.lo + gwarp) ? (t.hi - t.lo - gwarp + kWarpsPerGroup - 1) / kWarpsPerGroup : 0;
    return t;
  };
  auto no_more = []() {
    float4 e0, e1;
    Entry e{};
    e.b = -1;
    pack_entry(e, e0, e1);
    return e0;
  };

  // The team's next task through the mailbox (every thread).  Each use u is armed by
  // every member (expect 32 bytes) and filled by one send from the team's leader, who
  // takes a ticket and waits until its entry exists.
  uint32_t mb = 0;
  auto take_box = [&]() {
    if (first) mbar_expect_tx(&gs.mbar_box[mb & 1u], 32);
    if (leader) {
      float4 e0, e1 = make_float4(0.f, 0.f, 0.f, 0.f);
      const int r = resolve_ticket(P, qu, take_ticket(qu), e0, e1);
      if (r < 0) {
        if (r == -2) atomicOr(P.ws.error, 8u);
        e0 = no_more();
      }
      send_entry(gs, static_cast<int>(mb & 1u), e0, e1);
    }
    __syncwarp();
    if (group_any(group, !mbar_wait_cluster(&gs.mbar_box[mb & 1u], (mb >> 1) & 1u))) {
      if (first) atomicOr(P.ws.error, 2u);
      tm.ok = false;
    }
    const Entry e = unpack_entry(gs.mbox[mb & 1u][0], gs.mbox[mb & 1u][1]);
    ++mb;
    return e;
  };

  Entry cur = take_box();
  uint32_t t = 0;  // tasks done by this team
  // a drawn token still to be found by this member's first warp (at the next task's start)
  bool srch = false;
  int s_b = 0, s_J = 0, s_par = 0;
  float s_base = 0.f, s_target = 0.f;
  float s_m = 0.f, s_c = 0.f, s_invZ = 1.f;
  bool s_noq = true;

  while (cur.b >= 0 && tm.ok) {
    const int par = static_cast<int>(t & 1u);
    // the previous task's draw, if this member holds u * S (its masses stay put until the
    // barrier at the end of this task's chunks)
    if (srch && gwarp == 0) {
      const T* lrow = reinterpret_cast<const T*>(logits + (static_cast<int64_t>(s_b) * R + s_J) * row_bytes);
      const float* qrow = s_noq ? nullptr : P.q + (static_cast<int64_t>(s_b) * P.gamma + s_J) * V;
      const int y = local_search<T, kHost>(lrow, qrow, V, d0, d1 - d0, s_base, s_target, s_m, s_c, s_invZ, s_noq,
                                    gs.mass[s_par], lane);
      if (lane == 0) P.out_tokens[static_cast<int64_t>(s_b) * R + s_J] = y;
    }
    srch = false;

    const int b = cur.b, ri = cur.row, kind = cur.kind;
    const float Tc = cur.T;
    const bool greedy = P.greedy_only || is_greedy(Tc);
    const float c = greedy ? 0.f : kLog2e / Tc;
    const Task tc = make_task(cur);
    const int gb = gamma_of(b);
    const bool gbad = gb < 0 || gb > P.gamma;  // a count of drafts out of range

    // This task's inputs (first thread): the draft and the uniforms now, the logit and q at
    // the draft once the draft has arrived.
    const bool at_draft = kind == kTaskRow && !gbad && ri < gb;
    int gx = -1;
    float gu = 0.f, gug = 0.f, glx = 0.f, gqx = 0.f;
    bool g2 = false;
    if (first) {
      if (at_draft) gx = __ldg(P.drafts + static_cast<int64_t>(b) * P.gamma + ri);
      if (!P.greedy_only) {
        if (at_draft) gu = __ldg(P.u + static_cast<int64_t>(b) * R + ri);
        if (!gbad) gug = __ldg(P.u + static_cast<int64_t>(b) * R + gb);
      }
    }
    auto gather2 = [&]() {
      if (first && !g2) {
        g2 = true;
        if (at_draft && !P.greedy_only && gx >= 0 && gx < V) {
          glx = load_elem<kHost>(reinterpret_cast<const T*>(tc.src), gx);
          gqx = load_in<kHost>(P.q + (static_cast<int64_t>(b) * P.gamma + ri) * V + gx);
        }
      }
    };

    // This task's copies: kSeqStages in flight for a row (kSeqDrawStages for a draw), one
    // more as each stage is read.
    int ci = 0;
    auto refill = [&]() {
      if (pp.ok && ci < tc.n) issue_job<T, kHost>(pp, tc, ci++, gwarp, lane, V, row_bytes);
    };
    const uint32_t depth = (kind == kTaskRow || cur.deep) ? kSeqStages : kSeqDrawStages;
    while (pp.ok && ci < tc.n && pp.in_flight() < depth) issue_job<T, kHost>(pp, tc, ci++, gwarp, lane, V, row_bytes);

    float4 mine;
    if (kind == kTaskRow) {
      float ml = -kInf, Zl = 0.f;
      int zl = INT_MAX;
      for (int j = 0; j < tc.n && pp.ok; ++j) {
        if (!pp.wait()) {
          if (lane == 0) atomicOr(P.ws.error, 1u);
          pp.ok = false;
          break;
        }
        const int ch = c0 + gwarp + j * kWarpsPerGroup;
        const int nv = static_cast<int>(
            min(static_cast<int64_t>(kSeqChunkBytes), row_bytes - static_cast<int64_t>(ch) * kSeqChunkBytes) / 16);
        const uint4* vb = reinterpret_cast<const uint4*>(pp.stage(pp.k));
        uint4 w[VPL];
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
          const int e = lane + 32 * v;
          if (e < nv) {
            w[v] = vb[e];
          } else if constexpr (sizeof(T) == 2) {
            w[v] = make_uint4(kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2);
          } else {
            const uint32_t nf = __float_as_uint(-kInf);
            w[v] = make_uint4(nf, nf, nf, nf);
          }
        }
        __syncwarp();
        ++pp.k;
        refill();
        row_chunk<T>(w, nv, ch, greedy, c, lane, ml, Zl, zl);
        gather2();
      }
      gather2();
      RowSum r;
      r.m = ml;
      r.Z = Zl;
      r.z = zl;
      r = warp_merge(r, c);
      if (lane == 0) gs.wsum[gwarp] = r;
      group_sync(group);
      RowSum s;
      s.m = -kInf;
      s.Z = 0.f;
      s.z = INT_MAX;
      if (gwarp == 0) {
        if (lane < kWarpsPerGroup) s = gs.wsum[lane];
        s = warp_merge(s, c);
      }
      mine = make_float4(s.m, s.Z, __int_as_float(s.z), 0.f);
    } else {
      const float nmc = -__fmul_rn(cur.m, c), invZ = 1.f / cur.Z;
      const bool with_q = tc.q != nullptr;
      float qmx = 0.f, qmn = 0.f;
      for (int j = 0; j < tc.n && pp.ok; ++j) {
        if (!pp.wait()) {
          if (lane == 0) atomicOr(P.ws.error, 1u);
          pp.ok = false;
          break;
        }
        const int cd = d0 + gwarp + j * kWarpsPerGroup;
        const int ng = min(kSeqDrawChunk, V - cd * kSeqDrawChunk) / 4;
        const unsigned char* sbuf = pp.stage(pp.k);
        GL lw[GPL];
        float4 qv[GPL];
#pragma unroll
        for (int v = 0; v < GPL; ++v) {
          const int g = lane + 32 * v;
          if (g < ng) {
            lw[v] = reinterpret_cast<const GL*>(sbuf)[g];
            qv[v] = with_q ? reinterpret_cast<const float4*>(sbuf + LB)[g] : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        __syncwarp();
        ++pp.k;
        refill();
        float sr = 0.f;
#pragma unroll
        for (int v = 0; v < GPL; ++v) {
          if (lane + 32 * v < ng) {
            float w4[4];
            sr += group_weights<T>(lw[v], qv[v], nmc, c, invZ, !with_q, w4);
            qmx = max_nan(qmx, max_nan(max_nan(qv[v].x, qv[v].y), max_nan(qv[v].z, qv[v].w)));
            qmn = fminf(qmn, fminf(fminf(qv[v].x, qv[v].y), fminf(qv[v].z, qv[v].w)));
          }
        }
        sr = warp_sum(sr);
        if (lane == 0) gs.mass[par][cd - d0] = sr;
      }
      const bool qbad = group_any(group, !(qmx < kInf) || qmn < 0.f);  // also: every chunk mass is in place
      float tot = 0.f;
      if (gwarp == 0) tot = local_scan(gs.mass[par], d1 - d0, lane).total;
      mine = pack_total(tot, qbad ? 1 : 0, 0);
    }
    if (first) {  // this task's inputs for the decision
      int err = 0;
      if (at_draft) {
        if (gx < 0 || gx >= V) {
          err = SPECDEC_STATUS_BAD_TOKEN;
        } else if (!greedy) {
          if (!(gqx >= 0.f && gqx < kInf)) err |= SPECDEC_STATUS_BAD_PROB;
          if (!(gu >= 0.f && gu < 1.f)) err |= SPECDEC_STATUS_BAD_UNIFORM;
        }
      }
      float* g = gs.gq[par];
      g[0] = __int_as_float(gx);
      g[1] = glx;
      g[2] = gqx;
      g[3] = gu;
      g[4] = gug;
      g[5] = __int_as_float(err);
    }
    __syncwarp();
    const int xp = exchange(gs, tm, mine, group, gwarp, lane, P.ws.error);

    // The decision, taken by every thread on the same inputs.
    const float* g = gs.gq[par];
    int warn = cur.warn;  // status bits above the error byte, >> 8
    bool done = false, failed = false, drawn = false;
    int J = -1, y = -1, st = 0;
    bool nxt_local = false;  // the next task stays with this team (next row, second draw pass)
    Entry nxt = cur;
    if (kind == kTaskRow) {
      RowSum rs;
      {
        const float4 s0 = gs.slot[xp][0];
        rs.m = s0.x;
        rs.Z = s0.y;
        rs.z = __float_as_int(s0.z);
      }
#pragma unroll
      for (int r = 1; r < kC; ++r) {
        const float4 sr = gs.slot[xp][r];
        RowSum o;
        o.m = sr.x;
        o.Z = sr.y;
        o.z = __float_as_int(sr.z);
        rs = merge(rs, o, c);
      }
      int err = 0;
      if (gbad) err = SPECDEC_STATUS_BAD_TOKEN;
      else if (!P.greedy_only && !(Tc - Tc == 0.f)) err = SPECDEC_STATUS_BAD_TEMPERATURE;
      else if (!(rs.m == rs.m) || rs.m == kInf) err = SPECDEC_STATUS_BAD_LOGIT;
      else if (rs.m == -kInf) err = SPECDEC_STATUS_EMPTY_ROW;
      else if (at_draft) err = __float_as_int(g[5]);
      if (err) {
        st = err;
        done = failed = true;
      } else {
        bool acc = false;
        float pxi = kNaN;
        const int xi = __float_as_int(g[0]);
        if (at_draft) {
          if (greedy) {
            acc = (xi == rs.z);
          } else {
            pxi = ex2(fmaf(g[1], c, -__fmul_rn(rs.m, c))) / rs.Z;
            if (g[2] == 0.f) {
              warn |= SPECDEC_STATUS_ZERO_Q >> 8;
              acc = pxi > 0.f;
            } else {
              acc = g[3] * g[2] < pxi;
            }
          }
        }
        if (at_draft && leader && P.out_p_draft) P.out_p_draft[static_cast<int64_t>(b) * P.gamma + ri] = pxi;
        if (acc) {
          if (leader) P.out_tokens[static_cast<int64_t>(b) * R + ri] = xi;
          nxt_local = true;
          nxt.b = b;
          nxt.row = ri + 1;
          nxt.kind = kTaskRow;
          nxt.warn = warn;
          nxt.m = 0.f;
          nxt.Z = 1.f;
          nxt.T = Tc;
        } else {  // rejection at ri, or row gamma: the extra token comes from row ri
          J = ri;
          if (greedy) {
            y = rs.z;
            done = true;
          } else if (!(g[4] >= 0.f && g[4] < 1.f)) {
            st = SPECDEC_STATUS_BAD_UNIFORM;
            done = failed = true;
          } else {
            Entry e;  // the draw goes to the queue; any team may take it
            e.b = b;
            e.row = ri;
            e.kind = kTaskDraw;
            e.warn = warn;
            e.m = rs.m;
            e.Z = rs.Z;
            e.T = Tc;
            if (leader) publish_draw(qu, e);
          }
        }
      }
    } else {  // the members' totals of the drawn row
      J = ri;
      float S = 0.f;
      bool anybad = false;
#pragma unroll
      for (int r = 0; r < kC; ++r) {
        S += unpack_total(gs.slot[xp][r]);
        anybad |= __float_as_int(gs.slot[xp][r].z) != 0;
      }
      if (kind == kTaskDraw && anybad) {
        st = SPECDEC_STATUS_BAD_PROB;
        done = failed = true;
      } else if (kind == kTaskDraw && !(S > 0.f)) {
        // zero total residual (possible only through rounding): draw from p itself
        nxt_local = true;
        nxt = cur;
        nxt.kind = kTaskDrawP;
        nxt.warn = warn | (SPECDEC_STATUS_ZERO_RESIDUAL >> 8);
      } else {
        // the member whose part holds u * S (else the last member with mass) finds y
        const float target = g[4] * S;
        int rstar = -1, rlast = 0;
        float base = 0.f, run = 0.f, baselast = 0.f;
#pragma unroll
        for (int r = 0; r < kC; ++r) {
          const float tt = unpack_total(gs.slot[xp][r]);
          if (tt > 0.f) { rlast = r; baselast = run; }
          if (rstar < 0 && tt > 0.f && run + tt > target) { rstar = r; base = run; }
          run += tt;
        }
        if (rstar < 0) { rstar = rlast; base = baselast; }
        if (static_cast<int>(tm.rank) == rstar) {
          srch = true;
          s_b = b;
          s_J = J;
          s_par = par;
          s_base = base;
          s_target = target;
          s_m = cur.m;
          s_c = c;
          s_invZ = 1.f / cur.Z;
          s_noq = kind == kTaskDrawP || tc.q == nullptr;
        }
        done = drawn = true;
      }
    }
    if (done && tm.rank == 0 && gwarp == 0) {
      // outputs of a finished sequence (the drawn token is written by the member that finds it)
      const int Jo = failed ? -1 : J;
      if (lane < R) {
        if (failed || lane > Jo) P.out_tokens[static_cast<int64_t>(b) * R + lane] = -1;
        else if (lane == Jo && !drawn) P.out_tokens[static_cast<int64_t>(b) * R + lane] = y;
      }
      if (lane < P.gamma && P.out_p_draft && (failed || lane > Jo || lane >= gb || (greedy && lane >= Jo)))
        P.out_p_draft[static_cast<int64_t>(b) * P.gamma + lane] = kNaN;
      if (lane == 0) {
        P.out_J[b] = Jo;
        if (P.out_status) P.out_status[b] = st | (warn << 8);
        atomicAdd(qu.finished, 1u);
      }
    }
    // the next task: this sequence's next step, or new work through the mailbox
    cur = nxt_local ? nxt : take_box();
    ++t;
  }
  // a draw found in the last task
  if (srch && gwarp == 0 && tm.ok) {
    const T* lrow = reinterpret_cast<const T*>(logits + (static_cast<int64_t>(s_b) * R + s_J) * row_bytes);
    const float* qrow = s_noq ? nullptr : P.q + (static_cast<int64_t>(s_b) * P.gamma + s_J) * V;
    const int y = local_search<T, kHost>(lrow, qrow, V, d0, d1 - d0, s_base, s_target, s_m, s_c, s_invZ, s_noq,
                                  gs.mass[s_par], lane);
    if (lane == 0) P.out_tokens[static_cast<int64_t>(s_b) * R + s_J] = y;
  }
  // Copies still in flight (left by a bounded wait that gave up): wait for them, bounded,
  // before the CTA exits.
  if (lane == 0)
    for (; pp.k < pp.issued; ++pp.k) mbar_wait(pp.sbar(pp.k), (pp.k / kSeqStages) & 1u);
  // No CTA leaves while another member may still write into its shared memory.
  cluster_sync_all();
}

template <typename T, bool kHost>
cudaError_t launch_typed(const ChainParams& P, cudaStream_t stream) {
  constexpr int smem = kSeqWarps * kSeqStages * kSeqChunkBytes;
  static unsigned long long configured = 0;
  static int max_clusters[64] = {};
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  cudaLaunchConfig_t cfg{};
  cfg.blockDim = dim3(kSeqWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!(configured & bit)) {
    if (cudaError_t e = cudaFuncSetAttribute(chain_seq_kernel<T, kHost>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        e != cudaSuccess)
      return e;
    cfg.gridDim = dim3(static_cast<unsigned>(kC * device_sm_count()));
    int n = 0;
    if (cudaError_t e = cudaOccupancyMaxActiveClusters(&n, chain_seq_kernel<T, kHost>, &cfg); e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    max_clusters[dev & 63] = n;
    configured |= bit;
  }
  const int want = (P.B + kSeqGroups - 1) / kSeqGroups;
  const int clusters = min(max_clusters[dev & 63], want);
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * kC));
  return cudaLaunchKernelEx(&cfg, chain_seq_kernel<T, kHost>, P);
}

}  // namespace

cudaError_t launch_chain_seq(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream) {
  if (P.host_inputs) {
    if (ldt == SPECDEC_BF16) return launch_typed<uint16_t, true>(P, stream);
    return launch_typed<float, true>(P, stream);
  }
  if (ldt == SPECDEC_BF16) return launch_typed<uint16_t, false>(P, stream);
  return launch_typed<float, false>(P, stream);
}

}  // namespace specdec
