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
#include <type_traits>

#include "specdec_device.cuh"
#include "specdec_internal.h"

namespace specdec {

namespace {

constexpr uint32_t kNegInfBf16x2 = 0xFF80FF80u;
constexpr float kNaN = __builtin_nanf("");
constexpr int kWarpsPerGroup = kSeqWarps / kSeqGroups;
constexpr int kGroupThreads = kWarpsPerGroup * 32;
constexpr int kC = kSeqCluster;
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

__device__ __forceinline__ int warp_max_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ long long warp_incl_scan_ll(long long v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long n = __shfl_up_sync(0xffffffffu, v, o);
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

// Geometry of a draw task's copies: kElems elements of the drawn row per copy (logits at
// the stage's start, q at kLB), in kStages stages of kSeqDrawStageBytes that reuse a warp's
// row stages; each lane takes kGPL groups of 4 elements of a copy.
template <typename T> struct DrawGeo {
  static constexpr int kElems = sizeof(T) == 2 ? kSeqDrawElemsBf16 : kSeqDrawElemsF32;
  static constexpr int kLB = kElems * static_cast<int>(sizeof(T));
  static constexpr int kStages = kSeqStages * kSeqChunkBytes / kSeqDrawStageBytes;
  static constexpr int kGPL = kElems / 4 / 32;
  static_assert(kElems * (static_cast<int>(sizeof(T)) + 4) == kSeqDrawStageBytes, "logits and q fill a stage");
  static_assert(kStages >= 2, "two draw copies in flight per warp");
  static_assert(kElems % 128 == 0 && kLB % 16 == 0, "whole groups per lane, 16-byte copies");
};

// max(p - q, 0) with p = e * invZ, in one rounding (a saturating fused multiply-add; for a
// draft probability q >= 0 and p <= 1 the clamp at 1 never binds).
__device__ __forceinline__ float resid(float e, float invZ, float q) {
  float w;
  asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(w) : "f"(e), "f"(invZ), "f"(-q));
  return w;
}
// Three-input minimum (NaN ignored) and NaN-propagating maximum.
__device__ __forceinline__ float min3(float a, float b, float c) {
  float y;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
  float y;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

// Residual (or target) weights w of 4 consecutive elements: w_k = max(p_k - q_k, 0), p_k =
// 2^(l_k c - rnd(m_J c)) / Z (nmc = -rnd(m_J c)); q == 0 (the bonus row, or a zero
// residual) leaves p itself.  Returns the group's mass (w0 + w2) + (w1 + w3); the chunk
// masses and the final search both take this sum.
template <typename T>
__device__ __forceinline__ float group_weights(const typename Group<T>::L& lw, const float4& q4, float nmc,
                                               float c, float invZ, float (&w)[4]) {
  float l[4];
  Group<T>::unpack(lw, l);
  const unsigned long long c2 = f2pack(c, c), nmc2 = f2pack(nmc, nmc);
  float y0, y1, y2, y3;
  f2unpack(f2fma(f2pack(l[0], l[1]), c2, nmc2), y0, y1);
  f2unpack(f2fma(f2pack(l[2], l[3]), c2, nmc2), y2, y3);
  w[0] = resid(ex2(y0), invZ, q4.x);
  w[1] = resid(ex2(y1), invZ, q4.y);
  w[2] = resid(ex2(y2), invZ, q4.z);
  w[3] = resid(ex2(y3), invZ, q4.w);
  float s0, s1;
  f2unpack(f2add(f2pack(w[0], w[1]), f2pack(w[2], w[3])), s0, s1);
  return s0 + s1;
}

// Shared state of one group (one team member).  Its layout is the same in every CTA, so
// a member's slot in another CTA is this one's address mapped to that CTA.
struct GroupShared {
  float4 slot[2][kC];           // summary exchange slots by parity, one per member
  uint64_t xbar[2];             // their mbarriers
  float4 mbox[2][2];            // the next task's 32-byte entry, by task parity
  uint64_t mbar_box[2];         // their mbarriers
  RowSum wsum[kWarpsPerGroup];  // per-warp row summaries
  float4 ahead;                 // a row's statistics computed ahead, as read from the workspace
  // per task parity: draft token bits, its logit, its q, u_i, u_gamma, input error bits
  float gq[2][8];
  long long mass[2][kSeqMaxDrawChunks];  // draw: mass per chunk of this member's part (fixed point), by task parity
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

// One warp's bulk-copy pipeline in its kSeqStages * kSeqChunkBytes of shared memory: a
// row task cuts it into kSeqStages stages of kSeqChunkBytes, a draw task into
// DrawGeo<T>::kStages stages of kSeqDrawStageBytes.  Stage s completes on barrier s.  A
// task consumes every copy it issues, so the pipe is empty between tasks and each task
// starts its stages at 0 (begin()); `phase` keeps every barrier's parity across tasks.
struct Pipe {
  unsigned char* buf;
  uint64_t* bar;
  uint32_t k = 0, issued = 0;  // copies consumed and issued by the current task
  uint32_t phase = 0;          // bit s: parity of barrier s's next phase
  uint32_t si = 0, sk = 0;     // stages of the next copy to issue and to consume
  uint32_t nst = kSeqStages, sbytes = kSeqChunkBytes;
  bool ok = true;  // false once a bounded wait gave up

  __device__ __forceinline__ void begin(uint32_t stages, uint32_t stage_bytes) {
    nst = stages;
    sbytes = stage_bytes;
    k = issued = 0;
    si = sk = 0;
  }
  __device__ __forceinline__ unsigned char* stage(uint32_t s) { return buf + s * sbytes; }
  __device__ __forceinline__ unsigned char* cur() { return stage(sk); }
  __device__ __forceinline__ uint32_t in_flight() const { return issued - k; }
  // Issue one copy group (one or two copies) into the next stage: bulk copies by one lane,
  // or (kHost) 16-byte copies by every lane, each of which then arrives on the stage's
  // barrier.  The fence orders this warp's earlier reads of that stage (completed by a
  // __syncwarp) before the copy.
  template <bool kHost>
  __device__ __forceinline__ void issue(const void* a, uint32_t na, const void* b, uint32_t nb, int off_b, int lane) {
    uint64_t* br = bar + si;
    unsigned char* dst = stage(si);
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
    si = (si + 1 == nst) ? 0u : si + 1;
    ++issued;
  }
  // Wait for the oldest copy in flight; consume() then releases its stage.
  __device__ __forceinline__ bool wait() { return mbar_wait(bar + sk, (phase >> sk) & 1u); }
  __device__ __forceinline__ void consume() {
    phase ^= 1u << sk;
    sk = (sk + 1 == nst) ? 0u : sk + 1;
    ++k;
  }
};

// kTaskAhead: the statistics of a row that its chain's team will reach later, computed
// by a team that would otherwise wait for work and left in the workspace for the chain.
enum : int { kTaskRow = 1, kTaskDraw = 2, kTaskDrawP = 3, kTaskAhead = 4 };

// A task entry: 32 bytes, in the global rings and in a team's mailbox.
//   e0 = (sequence b (-1: no more work), row | kind << 8 | warnings << 16, m, Z)
//   e1 = (T, cached, 0, 0)
// (m, Z) are the drawn row's maximum and normaliser for draw tasks; the warnings are
// the sequence's status bits above the error byte, shifted down by 8; `cached` (draw
// tasks, host-resident logits) says that the drawn row's device copy is in place.
struct Entry {
  int b, row, kind, warn;
  float m, Z, T;
  int cached = 0;
};
__device__ __forceinline__ void pack_entry(const Entry& e, float4& e0, float4& e1) {
  e0 = make_float4(__int_as_float(e.b), __int_as_float(e.row | (e.kind << 8) | (e.warn << 16)), e.m, e.Z);
  e1 = make_float4(e.T, __int_as_float(e.cached), 0.f, 0.f);
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
  e.cached = __float_as_int(e1.y);
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
  int B, cap;
};
constexpr int kDrawTag = 1 << 30;

// A ticket for the team's next task.  `pre` is a start ticket the leader already took
// (UINT_MAX: none).  Once a start ticket comes back past the last sequence, the team
// (starts_left false) takes only draw tickets.
//
// Every sequence, the first ones too, is started through a ticket, by whichever team takes
// it: part of the grid may not be resident while other kernels hold SMs, and a sequence
// tied to a team that is not yet running would hold back every team that waits for the
// call to end.  So no team ever waits on a team that has not started.
__device__ __forceinline__ int take_ticket(const Queue& q, unsigned pre, bool& starts_left) {
  if (starts_left) {
    const unsigned s = pre != UINT_MAX ? pre : atomicAdd(q.start_ticket, 1u);
    if (s < static_cast<unsigned>(q.B)) return static_cast<int>(s);
    starts_left = false;
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
    if (d < q.cap && ld_acquire(q.ready_draws + d) != 0) {
      const float4* ent = q.ring_draws + 2 * static_cast<int64_t>(d);
      e0 = __ldcg(ent);
      e1 = __ldcg(ent + 1);
      return 1;
    }
    if (ld_relaxed(q.finished) >= static_cast<unsigned>(q.B)) return -1;
    if (t0 == 0) t0 = global_timer_ns();
    else if (global_timer_ns() - t0 > P.queue_wait_ns) return -2;
    __nanosleep(128);
  }
}

// (drop: the test hook that loses the publication, so that whoever takes the ticket waits
// until its bound gives up)
__device__ void publish_draw(const Queue& q, const Entry& e, bool drop) {
  float4 e0, e1;
  pack_entry(e, e0, e1);
  const unsigned k = atomicAdd(q.pub_draws, 1u);
  float4* ent = q.ring_draws + 2 * static_cast<int64_t>(k);
  __stcg(ent, e0);
  __stcg(ent + 1, e1);
  if (!drop) st_release(q.ready_draws + k, 1);
}

// Rows lo..hi of sequence b for teams that wait for work (one entry each, published in one
// batch).  The chain's team waits for their statistics instead of streaming them itself.
__device__ void publish_ahead(const Queue& q, int b, int lo, int hi, float T) {
  const unsigned k0 = atomicAdd(q.pub_draws, static_cast<unsigned>(hi - lo + 1));
  for (int r = lo; r <= hi; ++r) {
    const unsigned k = k0 + static_cast<unsigned>(r - lo);
    if (k >= static_cast<unsigned>(q.cap)) break;  // cannot happen: each row is published at most once
    Entry e;
    e.b = b;
    e.row = r;
    e.kind = kTaskAhead;
    e.warn = 0;
    e.m = 0.f;
    e.Z = 1.f;
    e.T = T;
    float4 e0, e1;
    pack_entry(e, e0, e1);
    float4* ent = q.ring_draws + 2 * static_cast<int64_t>(k);
    __stcg(ent, e0);
    __stcg(ent + 1, e1);
    st_release(q.ready_draws + k, 1);
  }
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
// draw, the q row; the member's chunk range [lo, hi) (4 KB chunks for a row,
// DrawGeo<T>::kElems-element chunks for a draw); this warp's jobs are the chunks
// lo + gwarp, lo + gwarp + W, ...
struct Task {
  int kind = 0;
  const char* src = nullptr;
  const float* q = nullptr;
  int lo = 0, hi = 0, n = 0;
};

template <typename T, bool kHost>
__device__ __forceinline__ void issue_job(Pipe& pp, const Task& t, int j, int gwarp, int lane, int V,
                                          int64_t row_bytes) {
  using DG = DrawGeo<T>;
  const int ch = t.lo + gwarp + j * kWarpsPerGroup;
  if (t.kind == kTaskRow) {
    const uint32_t nb = static_cast<uint32_t>(
        min(static_cast<int64_t>(kSeqChunkBytes), row_bytes - static_cast<int64_t>(ch) * kSeqChunkBytes));
    pp.issue<kHost>(t.src + static_cast<int64_t>(ch) * kSeqChunkBytes, nb, nullptr, 0, 0, lane);
  } else {
    const int n = min(DG::kElems, V - ch * DG::kElems);
    const int64_t off = static_cast<int64_t>(ch) * DG::kElems;
    pp.issue<kHost>(t.src + off * static_cast<int64_t>(sizeof(T)), static_cast<uint32_t>(n) * sizeof(T),
                    t.q ? t.q + off : nullptr, t.q ? static_cast<uint32_t>(n) * 4u : 0u, DG::kLB, lane);
  }
}

// One 4 KB chunk of a row into this lane's running (max, sum, argmax).
template <typename T>
__device__ __forceinline__ void row_chunk(const uint4 (&w)[kSeqChunkBytes / 512], int nv, int ch, bool greedy,
                                          float c, int lane, float& ml, float& Zl, int& zl) {
  constexpr int VEC = Vec<T>::n;
  constexpr int VPL = kSeqChunkBytes / 16 / 32;
  constexpr int EPC = kSeqChunkBytes / static_cast<int>(sizeof(T));
  // chunk maximum of this lane (bf16: per 16-byte vector first, kept for the argmax search)
  float mt;
  uint32_t mv[VPL];
  if constexpr (sizeof(T) == 2) {
#pragma unroll
    for (int j = 0; j < VPL; ++j) mv[j] = bf2max(bf2max(w[j].x, w[j].y), bf2max(w[j].z, w[j].w));
    uint32_t mm = mv[0];
#pragma unroll
    for (int j = 1; j < VPL; ++j) mm = bf2max(mm, mv[j]);
    mt = max_nan(bf16_lo(mm), bf16_hi(mm));
  } else {
    mt = -kInf;
#pragma unroll
    for (int j = 0; j < VPL; ++j)
      mt = max_nan(mt, max_nan(max_nan(__uint_as_float(w[j].x), __uint_as_float(w[j].y)),
                               max_nan(__uint_as_float(w[j].z), __uint_as_float(w[j].w))));
  }
  if (greedy) {
    // strictly larger maximum: locate its first index in this chunk (earlier chunks keep
    // ties).  Entries past the row's end hold -inf and never equal a larger maximum; a
    // NaN maximum matches nothing (the row is an input error).
    if (mt > ml || (mt != mt && ml == ml)) {
      int idx = INT_MAX;
      if (sizeof(T) == 2 && mt != 0.f) {
        // bf16: mt is one of the lane's values, so match its 16-bit pattern (zero is left to
        // the comparison below, where -0 and +0 are equal): the first 16-byte vector whose
        // per-vector maximum holds it, then the first half-word inside that vector
        const uint32_t p16 = __float_as_uint(mt) >> 16, pat = p16 | (p16 << 16);
        auto zero_half = [](uint32_t x) { return (x - 0x00010001u) & ~x & 0x80008000u; };
        int jv = VPL;
        uint4 hv = w[VPL - 1];
#pragma unroll
        for (int j = VPL - 1; j >= 0; --j) {
          if (zero_half(mv[j] ^ pat)) {
            jv = j;
            hv = w[j];
          }
        }
        if (jv < VPL) {
          const uint32_t ww[4] = {hv.x, hv.y, hv.z, hv.w};
          int e = VEC;
#pragma unroll
          for (int q = 3; q >= 0; --q) {
            const uint32_t z = zero_half(ww[q] ^ pat);  // the lowest set half is exact
            if (z) e = 2 * q + ((z & 0x8000u) ? 0 : 1);
          }
          if (e < VEC) idx = ch * EPC + (lane + 32 * jv) * VEC + e;
        }
      } else {
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
          const uint32_t ww[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            float v;
            if constexpr (sizeof(T) == 2) v = (e & 1) ? bf16_hi(ww[e >> 1]) : bf16_lo(ww[e >> 1]);
            else v = __uint_as_float(ww[e]);
            if (idx == INT_MAX && v == mt) idx = ch * EPC + (lane + 32 * j) * VEC + e;
          }
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

// The draw's running masses are exact sums in 64-bit fixed point, units of 2^-52 (every
// weight and mass is at most about 1): fp32 running sums would round at a few 1e-8 of S,
// and move draws whose uniform falls that close to a boundary of the CDF.  fx() is the one
// rounding, of each lane's fp32 sum of its weights in a chunk (mass pass) or of each
// weight (search) into these units.
__device__ __forceinline__ long long fx(float x) {
  // x >= 0 (weights and masses): x = m * 2^(e - 150) is m * 2^(e - 98) units, from the bits
  // with integer shifts (values below 2^-29 are truncated to whole units)
  const uint32_t b = __float_as_uint(x);
  const int e = static_cast<int>(b >> 23);
  const unsigned long long m = (b & 0x7FFFFFu) | (e ? 0x800000u : 0u);
  const int sh = (e ? e : 1) - 98;
  if (sh >= 0) return static_cast<long long>(m << sh);
  return sh > -64 ? static_cast<long long>(m >> -sh) : 0;
}
// u * S exactly, floored to the units (u in [0, 1) from its fp32 bits): for integer C,
// C > floor(u * S) holds exactly when C > u * S.
__device__ __forceinline__ long long fx_target(float u, long long S) {
  if (!(u > 0.f) || S <= 0) return 0;
  const uint32_t ub = __float_as_uint(u);
  const int e = static_cast<int>(ub >> 23);                 // biased exponent (u < 1: e <= 126)
  const unsigned long long m = e ? ((ub & 0x7FFFFFu) | 0x800000u) : (ub & 0x7FFFFFu);
  const int sh = 150 - (e ? e : 1);                          // u = m * 2^-sh, sh >= 24
  const unsigned long long us = static_cast<unsigned long long>(S);
  const unsigned long long lo = us * m, hi = __umul64hi(us, m);
  if (sh >= 128) return 0;
  if (sh >= 64) return static_cast<long long>(hi >> (sh - 64));
  return static_cast<long long>((lo >> sh) | (hi << (64 - sh)));
}

// Scan of this member's chunk masses (first warp): each lane sums a contiguous run of
// chunks.  The search repeats exactly this arithmetic, so the member's total and the
// search's running prefixes agree to the bit.
struct LocalScan {
  int c0, c1;
  long long mine, incl, total;
};
__device__ __forceinline__ LocalScan local_scan(const long long* mass, int n, int lane) {
  LocalScan s;
  const int cpl = (n + 31) / 32;
  s.c0 = min(lane * cpl, n);
  s.c1 = min(s.c0 + cpl, n);
  s.mine = 0;
  for (int q = s.c0; q < s.c1; ++q) s.mine += mass[q];
  s.incl = warp_incl_scan_ll(s.mine, lane);
  s.total = __shfl_sync(0xffffffffu, s.incl, 31);
  return s;
}

// Inverse-CDF search inside this member's part (first warp of the chosen member): the
// chunk whose running mass (from `base`, the mass of all earlier members) first exceeds
// `target`, then the element inside it.  If rounding leaves no such element, the last
// positive-weight element of the part is taken.
template <typename T, bool kHost>
__device__ int local_search(const T* lrow, const float* qrow, int V, int d0, int n, long long base, long long target,
                            float mJ, float c, float invZ, bool no_q, const long long* mass, int lane) {
  using GL = typename Group<T>::L;
  constexpr int GPL = DrawGeo<T>::kGPL;
  constexpr int CH = DrawGeo<T>::kElems;
  const LocalScan s = local_scan(mass, n, lane);
  int cstar = -1, lastpos = -1;
  long long cbase = 0, prelast = 0, pre = base + (s.incl - s.mine);
  for (int q = s.c0; q < s.c1; ++q) {
    const long long w = mass[q];
    if (w > 0) { lastpos = q; prelast = pre; }
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
  const int k0 = (d0 + cstar) * CH;
  const int ng = min(CH, V - k0) / 4;
  float w[GPL][4];
  long long gsum[GPL];  // a group's mass: the sum of its weights' units
  long long lane_tot = 0;
#pragma unroll
  for (int j = 0; j < GPL; ++j) {
    const int g = lane * GPL + j;
    gsum[j] = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) w[j][e] = 0.f;
    if (g < ng) {
      const GL lw = load_in<kHost>(reinterpret_cast<const GL*>(lrow + k0) + g);
      const float4 q4 = no_q ? make_float4(0.f, 0.f, 0.f, 0.f) : load_in<kHost>(reinterpret_cast<const float4*>(qrow + k0) + g);
      group_weights<T>(lw, q4, -__fmul_rn(mJ, c), c, invZ, w[j]);
#pragma unroll
      for (int e = 0; e < 4; ++e) gsum[j] += fx(w[j][e]);
      lane_tot += gsum[j];
    }
  }
  int last_pos = -1;
#pragma unroll
  for (int j = 0; j < GPL; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (w[j][e] > 0.f) last_pos = k0 + 4 * (lane * GPL + j) + e;
  const long long gincl = warp_incl_scan_ll(lane_tot, lane);
  const unsigned ghit = __ballot_sync(0xffffffffu, cbase + gincl > target);
  int y = -1;
  if (ghit) {
    const int fl = __ffs(ghit) - 1;
    if (lane == fl) {
      long long p2 = cbase + (gincl - lane_tot);
#pragma unroll
      for (int j = 0; j < GPL; ++j) {
        if (y < 0 && p2 + gsum[j] > target) {
          long long run = 0;
          int lastp = -1;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            run += fx(w[j][e]);
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

// A member's draw total (fixed point, as two words) and a bad-probability flag as one
// 16-byte exchange payload.
__device__ __forceinline__ float4 pack_total(long long t, int flag) {
  return make_float4(__int_as_float(static_cast<int>(t)), __int_as_float(static_cast<int>(t >> 32)),
                     __int_as_float(flag), 0.f);
}
__device__ __forceinline__ long long unpack_total(const float4& v) {
  return (static_cast<long long>(__float_as_int(v.y)) << 32) | static_cast<unsigned>(__float_as_int(v.x));
}

// ---------------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------------
template <typename T, bool kHost>
__global__ void __launch_bounds__(kSeqWarps * 32, 1) chain_seq_kernel(const ChainParams P) {
  using GL = typename Group<T>::L;
  constexpr int VPL = kSeqChunkBytes / 16 / 32;
  constexpr int GPL = DrawGeo<T>::kGPL;
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
  // The workspace counters are cleared by the kernel launched just before this one, which
  // lets this launch start early (programmatic dependent launch): wait for it here.
  grid_dependency_wait();

  const int R = P.gamma + 1;
  const int V = P.V;
  const int64_t row_bytes = static_cast<int64_t>(V) * sizeof(T);
  const int nch = static_cast<int>((row_bytes + kSeqChunkBytes - 1) / kSeqChunkBytes);
  const int nchd = (V + DrawGeo<T>::kElems - 1) / DrawGeo<T>::kElems;
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
  qu.cap = P.ws.ring_cap;

  // drafts to verify for sequence b: gamma, or its own count (the bonus row is row gb)
  auto gamma_of = [&](int b) { return P.gammas ? __ldg(P.gammas + b) : P.gamma; };
  auto make_task = [&](const Entry& e) {
    Task t;
    t.kind = e.kind == kTaskAhead ? kTaskRow : e.kind;
    t.src = logits + (static_cast<int64_t>(e.b) * R + e.row) * row_bytes;
    if constexpr (kHost)  // a drawn row whose device copy is in place: read it, not the host
      if (t.kind != kTaskRow && e.cached) t.src = P.row_cache + static_cast<int64_t>(e.b) * row_bytes;
    t.q = (e.kind == kTaskDraw && e.row < gamma_of(e.b)) ? P.q + (static_cast<int64_t>(e.b) * P.gamma + e.row) * V
                                                          : nullptr;
    t.lo = (t.kind == kTaskRow) ? c0 : d0;
    t.hi = (t.kind == kTaskRow) ? c1 : d1;
    t.n = (t.hi > t.lo + gwarp) ? (t.hi - t.lo - gwarp + kWarpsPerGroup - 1) / kWarpsPerGroup : 0;
    return t;
  };
  // The entry that ends a team's work: b = -1, or -2 when its wait for work gave up.
  auto no_more = [](int code) {
    float4 e0, e1;
    Entry e{};
    e.b = code;
    pack_entry(e, e0, e1);
    return e0;
  };

  // The team's next task through the mailbox (every thread).  Each use u is armed by
  // every member (expect 32 bytes) and filled by one send from the team's leader, who
  // takes a ticket and waits until its entry exists.
  uint32_t mb = 0;
  bool starts_left = true;  // (leader) start tickets may remain
  unsigned pre_ticket = UINT_MAX;  // (leader) a start ticket taken while publishing a draw
  auto take_box = [&]() {
    if (first) mbar_expect_tx(&gs.mbar_box[mb & 1u], 32);
    if (leader) {
      float4 e0, e1 = make_float4(0.f, 0.f, 0.f, 0.f);
      const int r = resolve_ticket(P, qu, take_ticket(qu, pre_ticket, starts_left), e0, e1);
      pre_ticket = UINT_MAX;
      if (r < 0) {
        if (r == -2) atomicOr(P.ws.error, 8u);
        e0 = no_more(r == -2 ? -2 : -1);
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
  // rows ahead_lo..ahead_hi of the team's current chain went to teams that waited for work
  int ahead_lo = INT_MAX, ahead_hi = -1;
  // every start ticket is taken, and teams wait for work (as the leader last reported the
  // queues; every thread holds both)
  bool starts_gone = false, teams_wait = false;
  // a drawn token for this member to find (its second warp, while the team takes a ticket)
  bool srch = false;
  int s_b = 0, s_J = 0, s_par = 0;
  long long s_base = 0, s_target = 0;
  float s_m = 0.f, s_c = 0.f, s_invZ = 1.f;
  bool s_noq = true, s_cached = false;

  while (cur.b >= 0 && tm.ok) {
    const int par = static_cast<int>(t & 1u);
    // the previous task's draw, if this member holds u * S (its masses stay put until the
    // barrier at the end of this task's chunks)

    const int b = cur.b, ri = cur.row, kind = cur.kind;
    const float Tc = cur.T;
    const bool greedy = P.greedy_only || is_greedy(Tc);
    const float c = greedy ? 0.f : kLog2e / Tc;
    // a row of this chain whose statistics another team computes: read, not streamed
    const bool ahead_row = kind == kTaskRow && ri >= ahead_lo && ri <= ahead_hi;
    Task tc = make_task(cur);
    if (ahead_row) tc.n = 0;
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
    // teams waiting for work, seen by the leader as its row starts (sent with its summary)
    unsigned w_dt = 0, w_pd = 0, w_st = 0;
    if (leader && kind == kTaskRow && !ahead_row) {
      w_dt = ld_relaxed(qu.draw_ticket);
      w_pd = ld_relaxed(qu.pub_draws);
      w_st = ld_relaxed(qu.start_ticket);
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

    // This task's copies: a copy in every stage (kSeqStages of 4 KB for a row, two of 6 KB
    // for a draw), one more as each stage is read.
    int ci = 0;
    auto refill = [&]() {
      if (pp.ok && ci < tc.n) issue_job<T, kHost>(pp, tc, ci++, gwarp, lane, V, row_bytes);
    };
    if (tc.kind == kTaskRow) pp.begin(kSeqStages, kSeqChunkBytes);
    else pp.begin(DrawGeo<T>::kStages, kSeqDrawStageBytes);
    // While every team is busy, a draw keeps one copy in flight per warp (rows keep a copy
    // in every stage), so the rows -- the chains, the critical path -- get the larger share
    // of the bandwidth; once teams wait for work, every stage.
    const uint32_t depth = (tc.kind == kTaskRow || teams_wait) ? pp.nst : 1u;
    while (pp.ok && ci < tc.n && pp.in_flight() < depth) issue_job<T, kHost>(pp, tc, ci++, gwarp, lane, V, row_bytes);

    float4 mine = make_float4(0.f, 0.f, 0.f, 0.f);
    bool ahead_fail = false;
    if (ahead_row) {
      // the statistics another team left in the workspace (each member reads them)
      gather2();
      if (first) {
        const int64_t hk = static_cast<int64_t>(b) * R + ri;
        uint64_t t0 = 0;
        bool got = true;
        while (ld_acquire(P.ws.help_ready + hk) == 0) {
          if (t0 == 0) t0 = global_timer_ns();
          else if (global_timer_ns() - t0 > kMaxWaitNs) { got = false; break; }
          __nanosleep(64);
        }
        if (got) gs.ahead = __ldcg(P.ws.help + hk);
        else atomicOr(P.ws.error, 16u);
        ahead_fail = !got;
      }
    } else if (tc.kind == kTaskRow) {
      float ml = -kInf, Zl = 0.f;
      int zl = INT_MAX;
      // host-resident logits: this chain's own row also goes to the sequence's device copy,
      // which a draw from this row then reads instead of the host (rows computed ahead for
      // another team's chain are not copied)
      const bool to_cache = kHost && P.row_cache != nullptr && kind == kTaskRow;
      for (int j = 0; j < tc.n && pp.ok; ++j) {
        if (!pp.wait()) {
          if (lane == 0) atomicOr(P.ws.error, 1u);
          pp.ok = false;
          break;
        }
        const int ch = c0 + gwarp + j * kWarpsPerGroup;
        const int nv = static_cast<int>(
            min(static_cast<int64_t>(kSeqChunkBytes), row_bytes - static_cast<int64_t>(ch) * kSeqChunkBytes) / 16);
        const uint4* vb = reinterpret_cast<const uint4*>(pp.cur());
        uint4 w[VPL];
        if (nv == VPL * 32) {  // a whole chunk
#pragma unroll
          for (int v = 0; v < VPL; ++v) w[v] = vb[lane + 32 * v];
        } else {  // the row's last chunk: -inf past its end
          constexpr uint32_t nf = sizeof(T) == 2 ? kNegInfBf16x2 : 0xFF800000u;
#pragma unroll
          for (int v = 0; v < VPL; ++v) w[v] = (lane + 32 * v < nv) ? vb[lane + 32 * v] : make_uint4(nf, nf, nf, nf);
        }
        __syncwarp();
        pp.consume();
        refill();
        if constexpr (kHost) {
          if (to_cache) {
            uint4* dst = reinterpret_cast<uint4*>(P.row_cache + static_cast<int64_t>(b) * row_bytes +
                                                  static_cast<int64_t>(ch) * kSeqChunkBytes);
#pragma unroll
            for (int v = 0; v < VPL; ++v)
              if (lane + 32 * v < nv) __stcg(dst + lane + 32 * v, w[v]);
          }
        }
        row_chunk<T>(w, nv, ch, greedy, c, lane, ml, Zl, zl);
        gather2();
      }
      gather2();
      // the copy is visible device-wide before this row's summary leaves the member (every
      // reader of the copy learns of the draw through that summary or after it)
      if (to_cache) __threadfence();
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
      // the leader's view of the queues: teams waiting for work, and whether start tickets
      // may remain (bit 30)
      const int idle = static_cast<int>(w_dt - w_pd);
      const bool starts_remain = leader && w_st < static_cast<unsigned>(P.B);
      const int qv = min(max(idle, 0), (1 << 30) - 1) | (starts_remain ? (1 << 30) : 0);
      // bit 31: a copy wait of this member gave up (its summary is incomplete)
      const bool lost = group_any(group, !pp.ok);
      mine = make_float4(s.m, s.Z, __int_as_float(s.z), __int_as_float(qv | (lost ? INT_MIN : 0)));
    } else {
      const float nmc = -__fmul_rn(cur.m, c), invZ = 1.f / cur.Z;
      float qmx = 0.f, qmn = 0.f;
      // the chunks of the drawn row, with or without a q row (the bonus row, or a draw
      // from p after a zero residual)
      auto chunks = [&](auto with_q_t) {
        constexpr bool kWithQ = decltype(with_q_t)::value;
        using DG = DrawGeo<T>;
        for (int j = 0; j < tc.n && pp.ok; ++j) {
          if (!pp.wait()) {
            if (lane == 0) atomicOr(P.ws.error, 1u);
            pp.ok = false;
            break;
          }
          const int cd = d0 + gwarp + j * kWarpsPerGroup;
          const int ng = min(DG::kElems, V - cd * DG::kElems) / 4;  // groups of 4 in this chunk
          const GL* lb = reinterpret_cast<const GL*>(pp.cur());
          const float4* qb = reinterpret_cast<const float4*>(pp.cur() + DG::kLB);
          GL lw[GPL];
          float4 qv[GPL];
          if (ng == DG::kElems / 4) {  // a whole chunk
#pragma unroll
            for (int v = 0; v < GPL; ++v) {
              lw[v] = lb[lane + 32 * v];
              qv[v] = kWithQ ? qb[lane + 32 * v] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
          } else {  // the row's last chunk: -inf logits (zero weight) past its end
#pragma unroll
            for (int v = 0; v < GPL; ++v) {
              const bool in = lane + 32 * v < ng;
              if constexpr (sizeof(T) == 2) lw[v] = in ? lb[lane + 32 * v] : GL{kNegInfBf16x2, kNegInfBf16x2};
              else lw[v] = in ? lb[lane + 32 * v] : GL{0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u};
              qv[v] = (kWithQ && in) ? qb[lane + 32 * v] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
          __syncwarp();
          pp.consume();
          refill();
          float sr = 0.f;
#pragma unroll
          for (int v = 0; v < GPL; ++v) {
            float w4[4];
            sr += group_weights<T>(lw[v], qv[v], nmc, c, invZ, w4);
            if constexpr (kWithQ) {
              qmx = max3_nan(qmx, qv[v].x, qv[v].y);
              qmx = max3_nan(qmx, qv[v].z, qv[v].w);
              qmn = min3(qmn, qv[v].x, qv[v].y);
              qmn = min3(qmn, qv[v].z, qv[v].w);
            }
          }
          // the chunk's mass: the lanes' fp32 sums, added exactly in fixed point
          long long sx = fx(sr);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) sx += __shfl_xor_sync(0xffffffffu, sx, o);
          if (lane == 0) gs.mass[par][cd - d0] = sx;
        }
      };
      if (tc.q != nullptr) chunks(std::true_type{});
      else chunks(std::false_type{});
      const bool qbad = group_any(group, !(qmx < kInf) || qmn < 0.f);  // also: every chunk mass is in place
      long long tot = 0;
      if (gwarp == 0) tot = local_scan(gs.mass[par], d1 - d0, lane).total;
      const bool lost = group_any(group, !pp.ok);  // a copy wait of this member gave up
      mine = pack_total(tot, (qbad ? 1 : 0) | (lost ? 2 : 0));
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
    int xp = 0;
    if (!ahead_row) {
      xp = exchange(gs, tm, mine, group, gwarp, lane, P.ws.error);
    } else if (group_any(group, ahead_fail)) {  // (also makes gs.ahead visible to the group)
      tm.ok = false;  // the bounded wait for the statistics gave up
    }

    // A copy wait of either member gave up (the task's data are incomplete), or a wait on
    // the exchange or on a row computed ahead did: the team stops here, writing nothing
    // for this sequence; the kernel's last CTA reports it as timed out.
    bool lost = !tm.ok;
    if (!ahead_row && (kind == kTaskRow || kind == kTaskAhead)) {
#pragma unroll
      for (int r = 0; r < kC; ++r) lost |= __float_as_int(gs.slot[xp][r].w) < 0;
    } else if (!ahead_row) {
#pragma unroll
      for (int r = 0; r < kC; ++r) lost |= (__float_as_int(gs.slot[xp][r].z) & 2) != 0;
    }
    if (lost) {
      tm.ok = false;
      break;
    }

    // The decision, taken by every thread on the same inputs.
    if (kind == kTaskRow && !ahead_row) {
      starts_gone = !(__float_as_int(gs.slot[xp][0].w) & (1 << 30));
      teams_wait = (__float_as_int(gs.slot[xp][0].w) & ((1 << 30) - 1)) > 0;
    }
    const float* g = gs.gq[par];
    int warn = cur.warn;  // status bits above the error byte, >> 8
    bool done = false, failed = false, drawn = false;
    int J = -1, y = -1, st = 0;
    bool nxt_local = false;  // the next task stays with this team (next row, second draw pass)
    Entry nxt = cur;
    // a row's statistics: the members' summaries merged in member order, or those read
    // from the workspace for a row computed ahead
    RowSum rs;
    if (ahead_row) {
      rs.m = gs.ahead.x;
      rs.Z = gs.ahead.y;
      rs.z = __float_as_int(gs.ahead.z);
    } else if (kind == kTaskRow || kind == kTaskAhead) {
      const float4 s0 = gs.slot[xp][0];
      rs.m = s0.x;
      rs.Z = s0.y;
      rs.z = __float_as_int(s0.z);
#pragma unroll
      for (int r = 1; r < kC; ++r) {
        const float4 sr = gs.slot[xp][r];
        RowSum o;
        o.m = sr.x;
        o.Z = sr.y;
        o.z = __float_as_int(sr.z);
        rs = merge(rs, o, c);
      }
    }
    if (kind == kTaskAhead) {
      // left for the chain's team, which waits on the flag
      if (leader) {
        const int64_t hk = static_cast<int64_t>(b) * R + ri;
        __stcg(P.ws.help + hk, make_float4(rs.m, rs.Z, __int_as_float(rs.z), 0.f));
        st_release(P.ws.help_ready + hk, 1);
      }
    } else if (kind == kTaskRow) {
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
          // Teams wait for work: hand them this chain's later rows (from ri + 2; this team
          // goes on with ri + 1), one row per waiting team.
          const int idle = ahead_row ? 0 : (__float_as_int(gs.slot[xp][0].w) & ((1 << 30) - 1));
          const int lo = max(ri + 2, ahead_hi + 1), hi = min(gb, ri + 1 + idle);
          if (idle > 0 && lo <= hi) {
            if (leader) publish_ahead(qu, b, lo, hi, Tc);
            ahead_lo = lo;
            ahead_hi = hi;
          }
        } else {  // rejection at ri, or row gamma: the extra token comes from row ri
          J = ri;
          if (greedy) {
            y = rs.z;
            done = true;
          } else if (!(g[4] >= 0.f && g[4] < 1.f)) {
            st = SPECDEC_STATUS_BAD_UNIFORM;
            done = failed = true;
          } else {
            Entry e;
            e.b = b;
            e.row = ri;
            e.kind = kTaskDraw;
            e.warn = warn;
            e.m = rs.m;
            e.Z = rs.Z;
            e.T = Tc;
            e.cached = (kHost && P.row_cache != nullptr && !ahead_row) ? 1 : 0;
            if (starts_gone) {
              // no sequence waits to start: this team draws now, while row J is in L2
              nxt_local = true;
              nxt = e;
            } else if (leader) {
              // the draw goes to the queue (any team may take it) so that this team starts
              // the next sequence; that start ticket's atomic goes out beside the
              // publication's
              if (starts_left) pre_ticket = atomicAdd(qu.start_ticket, 1u);
              publish_draw(qu, e, P.drop_draws != 0);
            }
          }
        }
      }
    } else {  // the members' totals of the drawn row
      J = ri;
      long long S = 0;
      bool anybad = false;
#pragma unroll
      for (int r = 0; r < kC; ++r) {
        S += unpack_total(gs.slot[xp][r]);
        anybad |= (__float_as_int(gs.slot[xp][r].z) & 1) != 0;
      }
      if (kind == kTaskDraw && anybad) {
        st = SPECDEC_STATUS_BAD_PROB;
        done = failed = true;
      } else if (kind == kTaskDraw && !(S > 0)) {
        // zero total residual (possible only through rounding): draw from p itself
        nxt_local = true;
        nxt = cur;
        nxt.kind = kTaskDrawP;
        nxt.warn = warn | (SPECDEC_STATUS_ZERO_RESIDUAL >> 8);
      } else {
        // the member whose part holds u * S (else the last member with mass) finds y
        const long long target = fx_target(g[4], S);
        int rstar = -1, rlast = 0;
        long long base = 0, run = 0, baselast = 0;
#pragma unroll
        for (int r = 0; r < kC; ++r) {
          const long long tt = unpack_total(gs.slot[xp][r]);
          if (tt > 0) { rlast = r; baselast = run; }
          if (rstar < 0 && tt > 0 && run + tt > target) { rstar = r; base = run; }
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
          s_cached = kHost && cur.cached != 0;
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
        if (!drawn) __stcg(P.ws.seq_done + b, 1);  // (a drawn token: once it is written)
        atomicAdd(qu.finished, 1u);
      }
    }
    // A draw ends its chain, so the team takes a ticket next: the member holding u * S
    // finds the drawn token with its second warp meanwhile (the leader, in the first warp,
    // fetches the ticket).
    if (srch && gwarp == 1) {
      const T* lrow = reinterpret_cast<const T*>(
          s_cached ? P.row_cache + static_cast<int64_t>(s_b) * row_bytes
                   : logits + (static_cast<int64_t>(s_b) * R + s_J) * row_bytes);
      const float* qrow = s_noq ? nullptr : P.q + (static_cast<int64_t>(s_b) * P.gamma + s_J) * V;
      const int y = local_search<T, kHost>(lrow, qrow, V, d0, d1 - d0, s_base, s_target, s_m, s_c, s_invZ, s_noq,
                                           gs.mass[s_par], lane);
      if (lane == 0) {
        P.out_tokens[static_cast<int64_t>(s_b) * R + s_J] = y;
        __stcg(P.ws.seq_done + s_b, 1);
      }
    }
    srch = false;
    // the next task: this sequence's next step, or new work through the mailbox
    if (!nxt_local) {
      ahead_lo = INT_MAX;
      ahead_hi = -1;
    }
    cur = nxt_local ? nxt : take_box();
    ++t;
  }
  // Copies still in flight (left by a bounded wait that gave up): wait for them, bounded,
  // before the CTA exits.
  if (lane == 0)
    for (; pp.k < pp.issued; pp.consume()) mbar_wait(pp.bar + pp.sk, (pp.phase >> pp.sk) & 1u);
  // A team whose wait gave up stopped with work left: sequences it (or the teams whose
  // work it was waiting for) did not finish.  Once every team has stopped this way -- then
  // no team is working -- the last one marks each sequence without its done flag as timed
  // out (J = -1, tokens -1, p_draft NaN).  Teams that ran out of work normally skip this.
  const bool abnormal = !tm.ok || cur.b == -2;

  // No CTA leaves while another member may still write into its shared memory.
  cluster_sync_all();

  if (abnormal && leader) {
    __threadfence();  // this team's outputs and done flags (its members: the cluster barrier)
    const unsigned teams = (gridDim.x / kC) * kSeqGroups;
    if (atomicAdd(P.ws.exit_count, 1u) == teams - 1) {
      __threadfence();
      for (int b = 0; b < P.B; ++b) {
        if (ld_acquire(P.ws.seq_done + b) != 0) continue;
        for (int i = 0; i < R; ++i) P.out_tokens[static_cast<int64_t>(b) * R + i] = -1;
        if (P.out_p_draft)
          for (int i = 0; i < P.gamma; ++i) P.out_p_draft[static_cast<int64_t>(b) * P.gamma + i] = kNaN;
        P.out_J[b] = -1;
        if (P.out_status) P.out_status[b] = SPECDEC_STATUS_TIMEOUT;
      }
    }
  }
}

// Clears the workspace's counter block (counters, flags and queue words that must start at
// zero) for the left-to-right kernel launched right after it, and lets that launch begin
// at once: its set-up overlaps this kernel, and it waits for this kernel before it uses
// the counters.
__global__ void __launch_bounds__(256) seq_clear_kernel(uint4* p, size_t n) {
  grid_launch_dependents();
  for (size_t i = threadIdx.x; i < n; i += blockDim.x) p[i] = make_uint4(0u, 0u, 0u, 0u);
}

template <typename T, bool kHost>
cudaError_t launch_typed(const ChainParams& P, cudaStream_t stream, bool pdl) {
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
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
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
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, chain_seq_kernel<T, kHost>, P);
}

}  // namespace

cudaError_t launch_chain_seq_clear(const ChainParams& P, cudaStream_t stream) {
  return launch_kernel(seq_clear_kernel, dim3(1), dim3(256), 0, stream, 0, reinterpret_cast<uint4*>(P.ws.error),
                       P.counter_bytes / 16);
}

cudaError_t launch_chain_seq(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream, bool pdl) {
  if (P.host_inputs) {
    if (ldt == SPECDEC_BF16) return launch_typed<uint16_t, true>(P, stream, pdl);
    return launch_typed<float, true>(P, stream, pdl);
  }
  if (ldt == SPECDEC_BF16) return launch_typed<uint16_t, false>(P, stream, pdl);
  return launch_typed<float, false>(P, stream, pdl);
}

}  // namespace specdec
