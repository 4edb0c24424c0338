// C-ABI entry points: argument validation, workspace layout, launches, kernel timing.

#include <atomic>
#include <cstdint>
#include <algorithm>
#include <mutex>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include <cuda_runtime.h>

#include "specdec.h"
#include "specdec_internal.h"

namespace specdec {

// Test hooks (specdec_set_test_hook): process-global, 0 = production behaviour.
std::atomic<int> g_test_hooks[SPECDEC_NUM_HOOKS];
int test_hook(int hook) { return (hook >= 0 && hook < SPECDEC_NUM_HOOKS) ? g_test_hooks[hook].load() : 0; }

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t elem_size(specdec_dtype t) { return t == SPECDEC_BF16 ? 2 : 4; }

bool valid_dtype(int t) { return t == SPECDEC_F32 || t == SPECDEC_BF16; }

// 16-byte vector loads need every row start 16-byte aligned.
bool rows_vectorizable(const void* base, int64_t V, size_t esize) {
  return aligned16(base) && ((V * static_cast<int64_t>(esize)) % 16 == 0);
}

// Aligned rows take the left-to-right kernel, which reads rows only up to the first
// rejection; the all-rows kernels serve them only under the test hook.
bool use_left_to_right() { return test_hook(SPECDEC_HOOK_CHAIN_ALL_ROWS) == 0; }

// Block verification runs as one launch that reads every row once; the statistics and
// mass kernels of the streaming path serve it only under the test hook.
bool block_two_pass() { return test_hook(SPECDEC_HOOK_BLOCK_TWO_PASS) != 0; }

// ---- last error (per host thread) -----------------------------------------------------
thread_local char g_last_error[256] = "no error";

int fail_cuda(const char* step, cudaError_t e) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", step, cudaGetErrorString(e),
                cudaGetErrorName(e));
  return SPECDEC_ERR_CUDA;
}
int fail(int code, const char* what) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s", what);
  return code;
}

// ---- kernel timing (process-global, single-threaded use) -----------------------------
struct ProfRecord {
  int kernel;
  cudaEvent_t start, stop;
};
bool g_prof_on = false;
std::vector<cudaEvent_t> g_prof_pool;
std::vector<ProfRecord> g_prof_records;
size_t g_prof_next = 0;

struct ProfScope {
  cudaStream_t stream;
  int kernel;
  bool active = false;
  ProfRecord rec{};
  ProfScope(int k, cudaStream_t s) : stream(s), kernel(k) {
    if (g_prof_on && g_prof_next + 2 <= g_prof_pool.size()) {
      rec = {k, g_prof_pool[g_prof_next], g_prof_pool[g_prof_next + 1]};
      g_prof_next += 2;
      active = cudaEventRecord(rec.start, stream) == cudaSuccess;
    }
  }
  ~ProfScope() {
    if (active && cudaEventRecord(rec.stop, stream) == cudaSuccess) g_prof_records.push_back(rec);
  }
};

}  // namespace

// Layout: [error word, draw count | arrival counters] -- the counter block, cleared on
// the stream at the start of every call -- then per-sequence state, the draw list, the
// per-segment (or per-chunk) summaries and the draw masses.  Returns the total bytes and
// the counter-block bytes (through counter_bytes when non-null).
size_t chain_workspace_layout(int B, int g, int V, specdec_dtype ldt, int path, void* base,
                              ChainWorkspace* ws, size_t* counter_bytes, bool block) {
  const int64_t rows = static_cast<int64_t>(B) * (g + 1);
  // drawn rows: one per sequence, or (block verification) every row's residual masses
  const int64_t n_drawn = block ? rows : static_cast<int64_t>(B);
  int64_t n_part, draw_bytes;
  if (path == 3) {  // single-read block verification: only the error word
    n_part = 0;
    draw_bytes = 0;
  } else if (path == 2) {
    const int64_t row_bytes = static_cast<int64_t>(V) * static_cast<int64_t>(elem_size(ldt));
    n_part = rows * ((row_bytes + kStatsChunkBytes - 1) / kStatsChunkBytes);
    draw_bytes = n_drawn * ((V + kDrawChunk - 1) / kDrawChunk) * static_cast<int64_t>(sizeof(float));
  } else {
    const int seg = chain_segment_len(ldt, path == 1);
    const int64_t nseg = (static_cast<int64_t>(V) + seg - 1) / seg;
    n_part = rows * nseg;
    draw_bytes = static_cast<int64_t>(B) * nseg * static_cast<int64_t>(sizeof(double2));
  }
  // queue entries of the left-to-right kernel (streaming layout only)
  const int64_t n_entries = path == 2 ? static_cast<int64_t>(B) * g + 2 * static_cast<int64_t>(B) : 0;
  // (the streaming layout also keeps a bad-draft-probability flag per sequence and, for
  // the left-to-right kernel, a ready flag per row for statistics computed ahead)
  const int64_t n_help = path == 2 ? rows : 0;
  const int64_t n_done = path == 2 ? B : 0;  // left-to-right kernel: sequence finished
  const int64_t n_counters = path == 3 ? 0
                                        : std::max<int64_t>(2 * static_cast<int64_t>(B),
                                                            n_entries + (path == 2 ? B : 0) + n_help + n_done);
  size_t off = 0;
  const size_t o_error = off;    off += kAlign;
  const size_t o_counters = off; off += round_up(sizeof(unsigned) * static_cast<size_t>(n_counters));
  const size_t counters_end = off;
  const size_t o_ring = off;     off += round_up(2 * sizeof(float4) * static_cast<size_t>(n_entries));
  const size_t o_help = off;     off += round_up(sizeof(float4) * static_cast<size_t>(n_help));
  const size_t o_seq = off;      off += round_up(sizeof(SeqState) * static_cast<size_t>(B));
  const size_t o_list = off;     off += round_up(sizeof(DrawEntry) * static_cast<size_t>(n_drawn));
  const size_t o_brows = off;    off += block ? round_up(sizeof(float4) * static_cast<size_t>(rows)) : 0;
  const size_t o_part = off;     off += round_up(sizeof(float4) * static_cast<size_t>(n_part));
  const size_t o_draw = off;     off += round_up(static_cast<size_t>(draw_bytes));
  if (counter_bytes) *counter_bytes = counters_end;
  if (base != nullptr && ws != nullptr) {
    char* p = static_cast<char*>(base);
    ws->error = reinterpret_cast<unsigned*>(p + o_error);
    ws->draw_count = reinterpret_cast<unsigned*>(p + o_error) + 1;
    ws->counters = reinterpret_cast<unsigned*>(p + o_counters);
    ws->seq = reinterpret_cast<SeqState*>(p + o_seq);
    ws->draw_list = reinterpret_cast<DrawEntry*>(p + o_list);
    ws->partials = reinterpret_cast<float4*>(p + o_part);
    ws->draw = reinterpret_cast<double2*>(p + o_draw);
    ws->draw_mass = reinterpret_cast<float*>(p + o_draw);
    ws->queue = reinterpret_cast<unsigned*>(p + o_error) + 2;
    ws->ready = reinterpret_cast<int*>(p + o_counters);
    ws->ring = reinterpret_cast<float4*>(p + o_ring);
    ws->qbad = path == 2 ? reinterpret_cast<int*>(p + o_counters) + n_entries : nullptr;
    ws->help_ready = path == 2 ? reinterpret_cast<int*>(p + o_counters) + n_entries + B : nullptr;
    ws->seq_done = path == 2 ? reinterpret_cast<int*>(p + o_counters) + n_entries + B + n_help : nullptr;
    ws->exit_count = reinterpret_cast<unsigned*>(p + o_error) + 6;
    ws->help = path == 2 ? reinterpret_cast<float4*>(p + o_help) : nullptr;
    ws->ring_cap = static_cast<int>(n_entries);
    ws->block_rows = block ? reinterpret_cast<float4*>(p + o_brows) : nullptr;

  }
  return off;
}

}  // namespace specdec

using namespace specdec;

namespace {

// Workspace sizing must not depend on pointer alignment, so size for the shorter
// (scalar-path) segment, which needs the most segments.
size_t chain_ws_bytes(int B, int g, int V, specdec_dtype ldt) {
  size_t m = 0;
  for (int path = 0; path < 3; ++path) {
    const size_t b = chain_workspace_layout(B, g, V, ldt, path, nullptr, nullptr, nullptr);
    m = b > m ? b : m;
  }
  return m;
}

bool chain_sizes_ok(int B, int g, int V) {
  if (B <= 0 || g <= 0 || V <= 0) return false;
  return true;
}

// The device copy of each sequence's latest row that the left-to-right kernel keeps when
// the logits sit in host memory (placed after the regular workspace).
size_t chain_row_cache_bytes(int B, int V, specdec_dtype ldt) {
  return round_up(static_cast<size_t>(B) * static_cast<size_t>(V) * elem_size(ldt));
}

int chain_common(const void* logits, specdec_dtype ldt, const float* q, const int32_t* drafts,
                 const float* temps, const float* u, int B, int g, int V, int32_t* out_tokens,
                 int32_t* out_J, float* out_p, int32_t* out_status, void* workspace,
                 size_t workspace_bytes, void* stream, bool greedy_only,
                 const int32_t* gammas = nullptr) {
  if (!valid_dtype(ldt)) return SPECDEC_ERR_INVALID_ARG;
  if (!chain_sizes_ok(B, g, V)) return SPECDEC_ERR_INVALID_ARG;
  if (!logits || !drafts || !out_tokens || !out_J || !workspace) return SPECDEC_ERR_INVALID_ARG;
  if (!greedy_only && (!q || !temps || !u)) return SPECDEC_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SPECDEC_ERR_INVALID_ARG;
  if (g > kMaxGamma) return SPECDEC_ERR_UNSUPPORTED;
  const size_t es = elem_size(ldt);
  bool vec = rows_vectorizable(logits, V, es);
  if (!greedy_only) vec = vec && rows_vectorizable(q, V, 4);
  // streaming path: aligned rows and a decision that fits one warp
  const bool stream_path = vec && (g + 1) <= kStreamMaxRows;
  const int seg = chain_segment_len(ldt, vec);
  const int64_t nseg = (static_cast<int64_t>(V) + seg - 1) / seg;
  const int64_t items = static_cast<int64_t>(B) * (g + 1) * nseg;
  if (items > INT32_MAX || nseg > 65535 || B > 65535) return SPECDEC_ERR_UNSUPPORTED;
  if (gammas && !(stream_path && V <= seq_max_v(ldt)))  // per-sequence counts: left-to-right kernel only
    return fail(SPECDEC_ERR_UNSUPPORTED, "per-sequence draft counts need 16-byte rows, g + 1 <= 32");
  if (workspace_bytes < chain_ws_bytes(B, g, V, ldt)) return SPECDEC_ERR_WORKSPACE;
  // logits and q in pinned host memory: the left-to-right kernel reads the rows it needs
  // over the host link; pageable host memory is refused (the first check that asks the
  // CUDA runtime)
  bool host_in = false, logits_on_host = false;
  for (const void* p : {logits, greedy_only ? nullptr : static_cast<const void*>(q)}) {
    if (p == nullptr) continue;
    cudaPointerAttributes a{};
    if (cudaError_t e = cudaPointerGetAttributes(&a, p); e != cudaSuccess) return fail_cuda("pointer attributes", e);
    if (a.type == cudaMemoryTypeUnregistered)
      return fail(SPECDEC_ERR_INVALID_ARG, "host logits and draft probabilities must be pinned (cudaHostAlloc, cudaHostRegister)");
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
      int cur = 0;
      if (cudaError_t e = cudaGetDevice(&cur); e != cudaSuccess) return fail_cuda("querying the current device", e);
      if (a.device != cur)
        return fail(SPECDEC_ERR_INVALID_ARG, "logits or draft probabilities on a device other than the current one");
    }
    if (a.type == cudaMemoryTypeHost) {
      if (a.devicePointer != p) return fail(SPECDEC_ERR_UNSUPPORTED, "host memory not mapped at its own address");
      host_in = true;
      logits_on_host |= p == logits;
    }
  }
  if (host_in && !(stream_path && (gammas || use_left_to_right()) && V <= seq_max_v(ldt)))
    return fail(SPECDEC_ERR_UNSUPPORTED,
                "host-resident logits or draft probabilities need the left-to-right kernel: 16-byte rows, g + 1 <= 32, "
                "V <= 1,048,576 (bf16) or 786,432 (fp32)");

  ChainParams P{};
  P.logits = logits;
  P.q = q;
  P.drafts = drafts;
  P.temps = greedy_only ? nullptr : temps;
  P.u = greedy_only ? nullptr : u;
  P.B = B;
  P.gamma = g;
  P.V = V;
  P.nseg = static_cast<int>(nseg);
  P.seg = seg;
  P.greedy_only = greedy_only ? 1 : 0;
  P.gammas = gammas;
  P.out_tokens = out_tokens;
  P.out_J = out_J;
  P.out_p_draft = greedy_only ? nullptr : out_p;
  P.out_status = out_status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int path = stream_path ? 2 : (vec ? 1 : 0);
  size_t counter_bytes = 0;
  chain_workspace_layout(B, g, V, ldt, path, workspace, &P.ws, &counter_bytes);
  // Arrival counters, queue words and flags must start at zero; other regions are always
  // written before they are read.  The left-to-right kernel's launch clears them itself
  // (a clearing kernel it overlaps); the other paths clear them here.
  const bool left_to_right = stream_path && (gammas || use_left_to_right()) && V <= seq_max_v(ldt);
  if (!left_to_right)
    if (cudaError_t e = cudaMemsetAsync(workspace, 0, counter_bytes, s); e != cudaSuccess)
      return fail_cuda("clearing the workspace counters", e);
  if (left_to_right) {
    P.counter_bytes = counter_bytes;
    P.grid_stats = device_sm_count();
    P.host_inputs = host_in ? 1 : 0;
    // host-resident logits and room for a device copy of each sequence's latest row: a
    // drawn row is then read from device memory, not a second time over the host link
    const size_t ws_base = chain_ws_bytes(B, g, V, ldt);
    if (logits_on_host && !greedy_only && workspace_bytes >= ws_base + chain_row_cache_bytes(B, V, ldt))
      P.row_cache = static_cast<char*>(workspace) + ws_base;
    P.drop_draws = test_hook(SPECDEC_HOOK_CHAIN_DROP_DRAWS) ? 1 : 0;
    const int wait_us = test_hook(SPECDEC_HOOK_QUEUE_WAIT_US);
    P.queue_wait_ns = wait_us > 0 ? static_cast<unsigned long long>(wait_us) * 1000ull : 1000000000ull;
    if (cudaError_t e = launch_chain_seq_clear(P, s); e != cudaSuccess) return fail_cuda("clearing the workspace counters", e);
    // (kernel timing brackets the kernel alone with events: no early start then)
    ProfScope prof(SPECDEC_KERNEL_CHAIN_SEQ, s);
    if (cudaError_t e = launch_chain_seq(P, ldt, s, !prof.active); e != cudaSuccess)
      return fail_cuda("left-to-right kernel", e);
    return SPECDEC_OK;
  }
  if (stream_path) {
    const int64_t row_bytes = static_cast<int64_t>(V) * static_cast<int64_t>(es);
    P.nch = static_cast<int>((row_bytes + kStatsChunkBytes - 1) / kStatsChunkBytes);
    P.nchd = (V + kDrawChunk - 1) / kDrawChunk;
    const int sms = device_sm_count();
    const int64_t stat_items = static_cast<int64_t>(B) * (g + 1) * P.nch;
    const int64_t draw_items = static_cast<int64_t>(B) * P.nchd;
    if (stat_items >= INT32_MAX || draw_items >= INT32_MAX) return SPECDEC_ERR_UNSUPPORTED;
    P.grid_stats = static_cast<int>(std::min<int64_t>(sms, (stat_items + kStatsWarps - 1) / kStatsWarps));
    P.grid_draw = static_cast<int>(std::min<int64_t>(sms, (draw_items + kDrawWarps - 1) / kDrawWarps));
    {
      ProfScope prof(SPECDEC_KERNEL_CHAIN_STATS, s);
      if (cudaError_t e = launch_chain_stream_stats(P, ldt, s); e != cudaSuccess) return fail_cuda("statistics kernel (streaming)", e);
    }
    {
      ProfScope prof(SPECDEC_KERNEL_CHAIN_DECIDE, s);
      if (cudaError_t e = launch_chain_stream_decide(P, ldt, s); e != cudaSuccess) return fail_cuda("decision kernel", e);
    }
    if (!greedy_only) {
      {
        ProfScope prof(SPECDEC_KERNEL_CHAIN_SAMPLE, s);
        if (cudaError_t e = launch_chain_stream_draw(P, ldt, s); e != cudaSuccess) return fail_cuda("draw kernel (streaming)", e);
      }
      ProfScope prof(SPECDEC_KERNEL_CHAIN_FINISH, s);
      if (cudaError_t e = launch_chain_stream_finish(P, ldt, s); e != cudaSuccess) return fail_cuda("finish kernel", e);
    }
    return SPECDEC_OK;
  }
  {
    ProfScope prof(SPECDEC_KERNEL_CHAIN_STATS, s);
    if (cudaError_t e = launch_chain_stats(P, ldt, vec, s); e != cudaSuccess) return fail_cuda("statistics kernel", e);
  }
  if (!greedy_only) {
    ProfScope prof(SPECDEC_KERNEL_CHAIN_SAMPLE, s);
    if (cudaError_t e = launch_chain_sample(P, ldt, vec, s); e != cudaSuccess) return fail_cuda("draw kernel", e);
  }
  return SPECDEC_OK;
}

// ---- built-in scratch for specdec_verify_chain_noalloc ---------------------------------
// One fixed array in device memory; every GPU that loads the library holds it until the
// process exits.  Host code must not pass the symbol itself to a kernel: its address in
// host code is a host-side stand-in.  The device address is looked up once per device and
// context: a device reset (cudaDeviceReset) makes a new primary context, which loads the
// module again, possibly at another address.
constexpr size_t kNoAllocScratchBytes = SPECDEC_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
void* g_scratch_ctx[kMaxDevices] = {};

// The driver's cuCtxGetCurrent (through the runtime's entry-point lookup, so the library
// needs no link to the driver library), or null where it is not available.
using CtxGetCurrent = int (*)(void**);
CtxGetCurrent ctx_get_current() {
  static const CtxGetCurrent fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<CtxGetCurrent>(nullptr);
    return reinterpret_cast<CtxGetCurrent>(f);
  }();
  return fn;
}

// Device address of the scratch array on the current device and context (looked up on the
// first use on each, and on every use where the context cannot be queried).
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return fail_cuda("querying the current device", e);
  if (dev < 0 || dev >= kMaxDevices) return fail(SPECDEC_ERR_UNSUPPORTED, "device index beyond the scratch table");
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  void* ctx = nullptr;
  const CtxGetCurrent get = ctx_get_current();
  const bool known = get != nullptr && get(&ctx) == 0 && ctx != nullptr;
  if (!known || g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    void* ptr = nullptr;
    if (cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch); e != cudaSuccess)
      return fail_cuda("looking up the built-in scratch array", e);
    if (!known) {  // cudaGetSymbolAddress made the context current: ask again
      ctx = nullptr;
      if (get == nullptr || get(&ctx) != 0) ctx = nullptr;
    }
    g_scratch_ptr[dev] = ptr;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return SPECDEC_OK;
}

}  // namespace

extern "C" {

size_t specdec_chain_workspace_bytes(int B, int g, int V, specdec_dtype ldt) {
  if (!valid_dtype(ldt) || !chain_sizes_ok(B, g, V)) return 0;
  return chain_ws_bytes(B, g, V, ldt);
}

size_t specdec_chain_host_workspace_bytes(int B, int g, int V, specdec_dtype ldt) {
  if (!valid_dtype(ldt) || !chain_sizes_ok(B, g, V)) return 0;
  return chain_ws_bytes(B, g, V, ldt) + chain_row_cache_bytes(B, V, ldt);
}

int specdec_verify_chain(const void* logits, specdec_dtype ldt, const float* draft_probs,
                         const int32_t* draft_tokens, const float* temperatures,
                         const float* uniforms, int B, int g, int V, int32_t* out_tokens,
                         int32_t* out_num_accepted, float* out_p_draft, int32_t* out_status,
                         void* workspace, size_t workspace_bytes, void* stream) {
  return chain_common(logits, ldt, draft_probs, draft_tokens, temperatures, uniforms, B, g, V,
                      out_tokens, out_num_accepted, out_p_draft, out_status, workspace,
                      workspace_bytes, stream, false);
}

int specdec_verify_chain_varlen(const void* logits, specdec_dtype ldt, const float* draft_probs,
                                const int32_t* draft_tokens, const float* temperatures,
                                const float* uniforms, const int32_t* gammas, int B, int g, int V,
                                int32_t* out_tokens, int32_t* out_num_accepted, float* out_p_draft,
                                int32_t* out_status, void* workspace, size_t workspace_bytes,
                                void* stream) {
  if (!gammas) return fail(SPECDEC_ERR_INVALID_ARG, "gammas is null");
  return chain_common(logits, ldt, draft_probs, draft_tokens, temperatures, uniforms, B, g, V, out_tokens,
                      out_num_accepted, out_p_draft, out_status, workspace, workspace_bytes, stream, false,
                      gammas);
}

size_t specdec_block_workspace_bytes(int B, int g, int V, specdec_dtype ldt) {
  if (!valid_dtype(ldt) || !chain_sizes_ok(B, g, V)) return 0;
  return std::max(chain_workspace_layout(B, g, V, ldt, 2, nullptr, nullptr, nullptr, true),
                  chain_workspace_layout(B, g, V, ldt, 3, nullptr, nullptr, nullptr, true));
}

int specdec_verify_block(const void* logits, specdec_dtype ldt, const float* draft_probs,
                         const int32_t* draft_tokens, const float* temperatures,
                         const float* uniforms, int B, int g, int V, int32_t* out_tokens,
                         int32_t* out_num_accepted, float* out_p_draft, int32_t* out_status,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (!valid_dtype(ldt)) return fail(SPECDEC_ERR_INVALID_ARG, "unknown logits dtype");
  if (!chain_sizes_ok(B, g, V)) return fail(SPECDEC_ERR_INVALID_ARG, "B, g and V must be positive");
  if (!logits || !draft_probs || !draft_tokens || !temperatures || !uniforms || !out_tokens ||
      !out_num_accepted || !workspace)
    return fail(SPECDEC_ERR_INVALID_ARG, "a required pointer is null");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(SPECDEC_ERR_INVALID_ARG, "the workspace must be 256-byte aligned");
  const size_t es = elem_size(ldt);
  if (!rows_vectorizable(logits, V, es) || !rows_vectorizable(draft_probs, V, 4) || g + 1 > kStreamMaxRows)
    return fail(SPECDEC_ERR_UNSUPPORTED, "block verification needs 16-byte aligned rows and g + 1 <= 32");
  if (workspace_bytes < specdec_block_workspace_bytes(B, g, V, ldt))
    return fail(SPECDEC_ERR_WORKSPACE, "workspace smaller than specdec_block_workspace_bytes");
  ChainParams P{};
  P.logits = logits;
  P.q = draft_probs;
  P.drafts = draft_tokens;
  P.temps = temperatures;
  P.u = uniforms;
  P.B = B;
  P.gamma = g;
  P.V = V;
  P.out_tokens = out_tokens;
  P.out_J = out_num_accepted;
  P.out_p_draft = out_p_draft;
  P.out_status = out_status;
  const int64_t row_bytes = static_cast<int64_t>(V) * static_cast<int64_t>(es);
  P.nch = static_cast<int>((row_bytes + kStatsChunkBytes - 1) / kStatsChunkBytes);
  P.nchd = (V + kDrawChunk - 1) / kDrawChunk;
  const int sms = device_sm_count();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  size_t counter_bytes = 0;
  if (!block_two_pass() && block_fused_fits(g, V, ldt)) {  // one launch; every row read once
    const int cm = block_mass_chunk(ldt);
    P.nchm = (V + cm - 1) / cm;
    chain_workspace_layout(B, g, V, ldt, 3, workspace, &P.ws, &counter_bytes, true);
    if (cudaError_t e = cudaMemsetAsync(workspace, 0, counter_bytes, s); e != cudaSuccess)
      return fail_cuda("clearing the workspace counters", e);
    ProfScope prof(SPECDEC_KERNEL_BLOCK_FUSED, s);
    if (cudaError_t e = launch_block_fused(P, ldt, s); e != cudaSuccess) return fail_cuda("block verification kernel", e);
    return SPECDEC_OK;
  }
  const int64_t stat_items = static_cast<int64_t>(B) * (g + 1) * P.nch;
  const int64_t draw_items = static_cast<int64_t>(B) * (g + 1) * P.nchd;
  if (stat_items >= INT32_MAX || draw_items >= INT32_MAX || B > 65535)
    return fail(SPECDEC_ERR_UNSUPPORTED, "too many rows for one call");
  P.grid_stats = static_cast<int>(std::min<int64_t>(sms, (stat_items + kStatsWarps - 1) / kStatsWarps));
  P.grid_draw = static_cast<int>(std::min<int64_t>(sms, (draw_items + kDrawWarps - 1) / kDrawWarps));
  chain_workspace_layout(B, g, V, ldt, 2, workspace, &P.ws, &counter_bytes, true);
  if (cudaError_t e = cudaMemsetAsync(workspace, 0, counter_bytes, s); e != cudaSuccess)
    return fail_cuda("clearing the workspace counters", e);
  {
    ProfScope prof(SPECDEC_KERNEL_CHAIN_STATS, s);
    if (cudaError_t e = launch_chain_stream_stats(P, ldt, s); e != cudaSuccess) return fail_cuda("statistics kernel (block)", e);
  }
  {
    ProfScope prof(SPECDEC_KERNEL_BLOCK_DECIDE, s);
    if (cudaError_t e = launch_block_decide(P, ldt, s); e != cudaSuccess) return fail_cuda("block decision kernel", e);
  }
  {
    ProfScope prof(SPECDEC_KERNEL_CHAIN_SAMPLE, s);
    if (cudaError_t e = launch_chain_stream_draw(P, ldt, s); e != cudaSuccess) return fail_cuda("mass kernel (block)", e);
  }
  ProfScope prof(SPECDEC_KERNEL_BLOCK_FINISH, s);
  if (cudaError_t e = launch_block_finish(P, ldt, s); e != cudaSuccess) return fail_cuda("block finish kernel", e);
  return SPECDEC_OK;
}

size_t specdec_greedy_workspace_bytes(int B, int g, int V, specdec_dtype ldt) {
  return specdec_chain_workspace_bytes(B, g, V, ldt);
}

int specdec_verify_greedy(const void* logits, specdec_dtype ldt, const int32_t* draft_tokens,
                          int B, int g, int V, int32_t* out_tokens, int32_t* out_num_accepted,
                          int32_t* out_status, void* workspace, size_t workspace_bytes,
                          void* stream) {
  return chain_common(logits, ldt, nullptr, draft_tokens, nullptr, nullptr, B, g, V, out_tokens,
                      out_num_accepted, nullptr, out_status, workspace, workspace_bytes, stream,
                      true);
}

size_t specdec_tree_workspace_bytes(int B, int N, int V, int max_depth, specdec_dtype ldt) {
  (void)B; (void)N; (void)V; (void)max_depth; (void)ldt;
  return 0;  // the walk keeps all of its state on chip
}

int specdec_verify_tree(const void* logits, specdec_dtype ldt, const int32_t* node_tokens,
                        const int32_t* parents, const float* temperatures, const float* uniforms,
                        int B, int N, int V, int max_depth, int32_t* out_tokens,
                        int32_t* out_path, int32_t* out_num_accepted, int32_t* out_status,
                        void* workspace, size_t workspace_bytes, void* stream) {
  (void)workspace; (void)workspace_bytes;
  if (!valid_dtype(ldt)) return SPECDEC_ERR_INVALID_ARG;
  if (B <= 0 || N < 0 || V <= 0 || max_depth < 1) return SPECDEC_ERR_INVALID_ARG;
  if (!logits || !temperatures || !uniforms || !out_tokens || !out_path || !out_num_accepted)
    return SPECDEC_ERR_INVALID_ARG;
  if (N > 0 && (!node_tokens || !parents)) return SPECDEC_ERR_INVALID_ARG;
  if (max_depth > kMaxTreeDepth || B > INT32_MAX) return SPECDEC_ERR_UNSUPPORTED;
  TreeParams P{};
  P.logits = logits;
  P.node_tokens = node_tokens;
  P.parents = parents;
  P.temps = temperatures;
  P.u = uniforms;
  P.B = B;
  P.N = N;
  P.V = V;
  P.D = max_depth;
  P.out_tokens = out_tokens;
  P.out_path = out_path;
  P.out_J = out_num_accepted;
  P.out_status = out_status;
  const bool vec = rows_vectorizable(logits, V, elem_size(ldt));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ProfScope prof(SPECDEC_KERNEL_TREE_WALK, s);
  if (cudaError_t e = launch_tree_walk(P, ldt, vec, s); e != cudaSuccess) return fail_cuda("tree walk kernel", e);
  return SPECDEC_OK;
}

int specdec_verify_tree_recursive(const void* logits, specdec_dtype ldt, const float* draft_probs,
                                  const int32_t* node_tokens, const int32_t* parents,
                                  const float* temperatures, const float* uniforms, int B, int N, int V,
                                  int max_depth, int flags, int32_t* out_tokens, int32_t* out_path,
                                  int32_t* out_num_accepted, int32_t* out_status, void* stream) {
  if (!valid_dtype(ldt)) return fail(SPECDEC_ERR_INVALID_ARG, "unknown logits dtype");
  if (B <= 0 || N < 0 || V <= 0 || max_depth < 1) return fail(SPECDEC_ERR_INVALID_ARG, "bad sizes");
  if (flags & ~SPECDEC_TREE_WITHOUT_REPLACEMENT) return fail(SPECDEC_ERR_INVALID_ARG, "unknown flag bits");
  if (!logits || !draft_probs || !temperatures || !uniforms || !out_tokens || !out_path || !out_num_accepted)
    return fail(SPECDEC_ERR_INVALID_ARG, "a required pointer is null");
  if (N > 0 && (!node_tokens || !parents)) return fail(SPECDEC_ERR_INVALID_ARG, "node tokens and parents needed");
  if (max_depth > kMaxTreeDepth) return fail(SPECDEC_ERR_UNSUPPORTED, "max_depth above 64");
  TreeParams P{};
  P.logits = logits;
  P.q = draft_probs;
  P.node_tokens = node_tokens;
  P.parents = parents;
  P.temps = temperatures;
  P.u = uniforms;
  P.B = B;
  P.N = N;
  P.V = V;
  P.D = max_depth;
  P.out_tokens = out_tokens;
  P.out_path = out_path;
  P.out_J = out_num_accepted;
  P.out_status = out_status;
  P.wor = (flags & SPECDEC_TREE_WITHOUT_REPLACEMENT) ? 1 : 0;
  const bool vec = rows_vectorizable(logits, V, elem_size(ldt)) && rows_vectorizable(draft_probs, V, 4);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ProfScope prof(SPECDEC_KERNEL_TREE_RR, s);
  // 16-byte rows: each row split across a cluster (tree_rr_cluster.cu); else one CTA per sequence
  const int C = vec ? tree_rr_cluster_size(B, V, ldt) : 0;
  cudaError_t e = C > 0 ? launch_tree_rr_cluster(P, ldt, C, s) : launch_tree_rr(P, ldt, vec, s);
  if (e != cudaSuccess) return fail_cuda("tree recursive-rejection kernel", e);
  return SPECDEC_OK;
}

namespace {
bool gumbel_vec(const void* p, int V, size_t es) { return rows_vectorizable(p, V, es); }
}  // namespace

size_t specdec_gumbel_workspace_bytes(int B, int g) {
  if (B <= 0 || g <= 0) return 0;
  return gumbel_workspace_bytes(B);
}

int specdec_verify_gumbel(const void* logits, specdec_dtype ldt, const int32_t* draft_tokens,
                          const float* temperatures, uint64_t seed, int B, int g, int V,
                          int32_t* out_tokens, int32_t* out_num_accepted, int32_t* out_status,
                          void* workspace, size_t workspace_bytes, void* stream) {
  if (!valid_dtype(ldt)) return fail(SPECDEC_ERR_INVALID_ARG, "unknown logits dtype");
  if (!chain_sizes_ok(B, g, V)) return fail(SPECDEC_ERR_INVALID_ARG, "B, g and V must be positive");
  if (!logits || !draft_tokens || !temperatures || !out_tokens || !out_num_accepted || !workspace)
    return fail(SPECDEC_ERR_INVALID_ARG, "a required pointer is null");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(SPECDEC_ERR_INVALID_ARG, "the workspace must be 256-byte aligned");
  if (g + 1 > 512 || B > 65535) return fail(SPECDEC_ERR_UNSUPPORTED, "g + 1 above 512 or B above 65535");
  if (workspace_bytes < gumbel_workspace_bytes(B))
    return fail(SPECDEC_ERR_WORKSPACE, "workspace smaller than specdec_gumbel_workspace_bytes");
  GumbelParams P{};
  P.logits = logits;
  P.drafts = draft_tokens;
  P.temps = temperatures;
  P.key0 = static_cast<uint32_t>(seed);
  P.key1 = static_cast<uint32_t>(seed >> 32);
  P.B = B;
  P.G = g;
  P.V = V;
  P.parts = gumbel_parts(B);
  P.out_tokens = out_tokens;
  P.out_J = out_num_accepted;
  P.out_status = out_status;
  const size_t state_bytes = (static_cast<size_t>(B) * sizeof(int) + 255) / 256 * 256;
  P.state = static_cast<int*>(workspace);
  P.partials = static_cast<char*>(workspace) + state_bytes;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaError_t e = cudaMemsetAsync(workspace, 0, state_bytes, s); e != cudaSuccess)
    return fail_cuda("clearing the workspace", e);
  ProfScope prof(SPECDEC_KERNEL_GUMBEL, s);
  if (cudaError_t e = launch_gumbel_verify(P, ldt, gumbel_vec(logits, V, elem_size(ldt)), s); e != cudaSuccess)
    return fail_cuda("Gumbel verification kernels", e);
  return SPECDEC_OK;
}

int specdec_gumbel_draft(const float* draft_probs, uint64_t seed, int B, int g, int V,
                         int32_t* out_draft_tokens, void* stream) {
  if (!chain_sizes_ok(B, g, V)) return fail(SPECDEC_ERR_INVALID_ARG, "B, g and V must be positive");
  if (!draft_probs || !out_draft_tokens) return fail(SPECDEC_ERR_INVALID_ARG, "a required pointer is null");
  if (static_cast<int64_t>(B) * g > INT32_MAX) return fail(SPECDEC_ERR_UNSUPPORTED, "too many rows");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ProfScope prof(SPECDEC_KERNEL_GUMBEL_DRAFT, s);
  if (cudaError_t e = launch_gumbel_draft(draft_probs, seed, B, g, V, gumbel_vec(draft_probs, V, 4),
                                          out_draft_tokens, s);
      e != cudaSuccess)
    return fail_cuda("Gumbel draft kernel", e);
  return SPECDEC_OK;
}

int specdec_gumbel_noise(uint64_t seed, int B, int rows, int V, float* out_noise, void* stream) {
  if (B <= 0 || rows <= 0 || V <= 0) return fail(SPECDEC_ERR_INVALID_ARG, "B, rows and V must be positive");
  if (!out_noise) return fail(SPECDEC_ERR_INVALID_ARG, "a required pointer is null");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaError_t e = launch_gumbel_noise(seed, B, rows, V, out_noise, s); e != cudaSuccess)
    return fail_cuda("Gumbel noise kernel", e);
  return SPECDEC_OK;
}

int specdec_compact_kv(void* cache, int64_t row_bytes, int64_t slot_stride, int64_t seq_stride,
                       int64_t num_slots, const int32_t* block_table, int block_size, int max_blocks,
                       int64_t block_stride, int B, const int32_t* prefix_len, const int32_t* path,
                       int max_depth, const int32_t* num_accepted, int32_t* out_new_len,
                       int32_t* out_status, void* stream) {
  if (!cache || !prefix_len || !path || !num_accepted) return fail(SPECDEC_ERR_INVALID_ARG, "a required pointer is null");
  if (B <= 0 || B > 65535 || max_depth < 1 || row_bytes <= 0 || slot_stride < row_bytes)
    return fail(SPECDEC_ERR_INVALID_ARG, "bad sizes");
  if (block_table && (block_size <= 0 || max_blocks <= 0 || block_stride < static_cast<int64_t>(block_size) * slot_stride))
    return fail(SPECDEC_ERR_INVALID_ARG, "bad paged layout");
  if (!block_table && (num_slots <= 0 || (B > 1 && seq_stride < num_slots * slot_stride)))
    return fail(SPECDEC_ERR_INVALID_ARG, "bad contiguous layout");
  KvCompactParams P{};
  P.base = static_cast<char*>(cache);
  P.row_bytes = row_bytes;
  P.slot_stride = slot_stride;
  P.seq_stride = seq_stride;
  P.block_stride = block_stride;
  P.num_slots = block_table ? static_cast<int64_t>(max_blocks) * block_size : num_slots;
  P.block_table = block_table;
  P.block_size = block_size;
  P.max_blocks = max_blocks;
  P.B = B;
  P.max_depth = max_depth;
  P.prefix_len = prefix_len;
  P.path = path;
  P.num_accepted = num_accepted;
  P.out_new_len = out_new_len;
  P.out_status = out_status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ProfScope prof(SPECDEC_KERNEL_KV_COMPACT, s);
  if (cudaError_t e = launch_kv_compact(P, s); e != cudaSuccess) return fail_cuda("KV compaction kernel", e);
  return SPECDEC_OK;
}

int specdec_build_tree_mask(const int32_t* parents, int N, int prefix_len, uint8_t* out_mask,
                            int64_t* out_position_ids, int32_t* out_depth, int32_t* out_status,
                            void* stream) {
  if (!parents || !out_mask || !out_position_ids || !out_status) return SPECDEC_ERR_INVALID_ARG;
  if (N <= 0 || prefix_len < 0) return SPECDEC_ERR_INVALID_ARG;
  if ((static_cast<int64_t>(prefix_len) + N) * N >= INT32_MAX) return SPECDEC_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ProfScope prof(SPECDEC_KERNEL_TREE_MASK, s);
  if (cudaError_t e = launch_tree_mask(parents, N, prefix_len, out_mask, out_position_ids, out_depth,
                                       out_status, s);
      e != cudaSuccess)
    return fail_cuda("tree mask kernel", e);
  return SPECDEC_OK;
}

int specdec_profile_start(int max_launches) {
  if (max_launches <= 0) return SPECDEC_ERR_INVALID_ARG;
  specdec_profile_stop();
  g_prof_pool.resize(static_cast<size_t>(max_launches) * 2);
  for (auto& e : g_prof_pool) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      e = nullptr;
      specdec_profile_stop();
      return SPECDEC_ERR_CUDA;
    }
  }
  g_prof_records.clear();
  g_prof_next = 0;
  g_prof_on = true;
  return SPECDEC_OK;
}

int specdec_profile_read(double* total_ms, int* launches, int n) {
  if (!total_ms || !launches || n <= 0) return SPECDEC_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) { total_ms[i] = 0.0; launches[i] = 0; }
  for (const auto& r : g_prof_records) {
    if (cudaEventSynchronize(r.stop) != cudaSuccess) return SPECDEC_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) return SPECDEC_ERR_CUDA;
    if (r.kernel >= 0 && r.kernel < n) { total_ms[r.kernel] += ms; launches[r.kernel] += 1; }
  }
  g_prof_records.clear();
  g_prof_next = 0;
  return SPECDEC_OK;
}

int specdec_profile_stop(void) {
  g_prof_on = false;
  for (auto& e : g_prof_pool)
    if (e) cudaEventDestroy(e);
  g_prof_pool.clear();
  g_prof_records.clear();
  g_prof_next = 0;
  return SPECDEC_OK;
}

const char* specdec_version(void) { return "0.3.0"; }

int specdec_set_test_hook(int hook, int value) {
  if (hook < 0 || hook >= SPECDEC_NUM_HOOKS) return SPECDEC_ERR_INVALID_ARG;
  if (value < 0) return SPECDEC_ERR_INVALID_ARG;
  if (hook == SPECDEC_HOOK_TREE_CLUSTER && !(value == 0 || value == 1 || value == 2 || value == 4 || value == 8))
    return SPECDEC_ERR_INVALID_ARG;
  if ((hook == SPECDEC_HOOK_CHAIN_ALL_ROWS || hook == SPECDEC_HOOK_BLOCK_TWO_PASS ||
       hook == SPECDEC_HOOK_CHAIN_DROP_DRAWS) && value > 1)
    return SPECDEC_ERR_INVALID_ARG;
  g_test_hooks[hook].store(value);
  return SPECDEC_OK;
}

int specdec_get_test_hook(int hook) { return test_hook(hook); }

const char* specdec_last_error(void) { return g_last_error; }

int specdec_verify_chain_noalloc(const void* logits, specdec_dtype ldt, const float* draft_probs,
                                 const int32_t* draft_tokens, const float* temperatures,
                                 const float* uniforms, int B, int g, int V, int32_t* out_tokens,
                                 int32_t* out_num_accepted, float* out_p_draft, int32_t* out_status,
                                 void* stream) {
  if (!valid_dtype(ldt) || !chain_sizes_ok(B, g, V)) return fail(SPECDEC_ERR_INVALID_ARG, "invalid dtype or size");
  const size_t need = chain_ws_bytes(B, g, V, ldt);
  if (need > kNoAllocScratchBytes) {
    std::snprintf(g_last_error, sizeof(g_last_error),
                  "specdec_verify_chain_noalloc: this shape needs %zu bytes of scratch; the built-in "
                  "scratch holds %zu bytes (use specdec_verify_chain with a caller workspace)",
                  need, kNoAllocScratchBytes);
    return SPECDEC_ERR_TOO_LARGE;
  }
  void* scratch = nullptr;
  if (int rc = noalloc_scratch(&scratch); rc != SPECDEC_OK) return rc;
  // chain_common clears the counters it relies on, on this stream, before any kernel runs.
  return chain_common(logits, ldt, draft_probs, draft_tokens, temperatures, uniforms, B, g, V,
                      out_tokens, out_num_accepted, out_p_draft, out_status, scratch,
                      kNoAllocScratchBytes, stream, false);
}

}  // extern "C"
