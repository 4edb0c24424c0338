// Host/device interface between the C-ABI layer and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "specdec.h"

namespace specdec {

// The value of a test hook (SPECDEC_HOOK_*, specdec_set_test_hook); 0 = production.
int test_hook(int hook);

constexpr int kChainThreads = 256;
constexpr int kChainVectorsPerThread = 8;    // 16-byte vectors per thread per segment
constexpr int kScalarElemsPerThread = 32;    // elements per thread per segment (scalar path)
constexpr int kMaxGamma = 255;               // drafts per sequence handled by one decision CTA
constexpr int kTreeThreads = 512;
constexpr int kMaxTreeDepth = 64;
constexpr int kTreeStageBytes = 200 * 1024;  // a node's logits + q rows staged in shared memory

// Per-sequence state handed from the decision step to the draw step.
struct SeqState {
  int4 meta;   // (J, mode, status, 0); mode 0: done, 1: draw from residual or bonus row
  float4 row;  // (row max m, normaliser Z, c = log2(e)/T, uniform of the extra token)
};

// A sequence that draws an extra token: its drawn row and that row's softmax constants,
// written by the decision kernel in one 32-byte record so a draw work item needs one load.
struct DrawEntry {
  int4 loc;    // (sequence b, drawn row J, 0, 0)
  float4 row;  // (row max m, c = log2(e)/T, 1/Z, 0)
};

struct ChainWorkspace {
  float4* partials;   // [B*(g+1)*nseg]: per segment (max, sum of 2^((l-max)c), argmax bits, 0)
  unsigned* counters; // [2B]: arrivals per sequence for the statistics and the draw kernels
  SeqState* seq;      // [B]
  double2* draw;      // [B*nseg]: per segment (residual mass, target mass) of the drawn row
  // streaming path only
  struct DrawEntry* draw_list;  // [B]: every sequence that draws an extra token, in any order
  unsigned* draw_count;  // [1]: entries in draw_list
  float* draw_mass;      // [B*nchd]: residual (or bonus) mass per chunk of the drawn row
  unsigned* error;       // [1]: set when a bounded wait gave up
  int* qbad;             // [B]: a bad draft probability met by the mass pass; cleared per call
  float4* block_rows;    // [B*(g+1)]: block verification's (m, Z, w_k, w_k / Z) per row

  // left-to-right kernel: the task queues and the statistics of rows computed ahead
  unsigned* queue;       // [4]: starts taken, entries published, entries claimed, sequences finished
  int* ready;            // [ring_cap]: entry published; cleared per call
  float4* ring;          // [2 * ring_cap]: 32-byte task entries (draws and rows computed ahead)
  int ring_cap;          // B*g + 2B
  float4* help;          // [B*(g+1)]: (m, Z, argmax bits, 0) of a row computed ahead for its chain
  int* help_ready;       // [B*(g+1)]: that row's statistics are in place; cleared per call
  int* seq_done;         // [B]: the sequence's outputs are written; cleared per call
  unsigned* exit_count;  // [1]: CTAs that finished; cleared per call
};

// Streaming (bulk-copy) path geometry.
#ifndef SPECDEC_STATS_WARPS
#define SPECDEC_STATS_WARPS 16
#endif
#ifndef SPECDEC_STATS_STAGES
#define SPECDEC_STATS_STAGES 3
#endif
#ifndef SPECDEC_STATS_CHUNK
#define SPECDEC_STATS_CHUNK 4096
#endif
#ifndef SPECDEC_DRAW_WARPS
#define SPECDEC_DRAW_WARPS 16
#endif
#ifndef SPECDEC_DRAW_STAGES
#define SPECDEC_DRAW_STAGES 4
#endif
#ifndef SPECDEC_DRAW_CHUNK
#define SPECDEC_DRAW_CHUNK 512
#endif
constexpr int kStatsWarps = SPECDEC_STATS_WARPS;     // warps per CTA, one CTA per SM
constexpr int kStatsStages = SPECDEC_STATS_STAGES;   // bulk-copy stages per warp
constexpr int kStatsChunkBytes = SPECDEC_STATS_CHUNK;
constexpr int kDrawWarps = SPECDEC_DRAW_WARPS;
constexpr int kDrawStages = SPECDEC_DRAW_STAGES;       // for bf16 logits
constexpr int kDrawStagesF32 = 3;                      // fp32 stages are larger
constexpr int kDrawChunk = SPECDEC_DRAW_CHUNK;       // elements of the drawn row per work item
constexpr int kStreamMaxRows = 32;    // gamma + 1 handled by one warp's decision

// Left-to-right (early-exit) kernel geometry.  One CTA per SM holds kSeqGroups groups of
// warps; a team is one group in each of the kSeqCluster CTAs of a thread-block cluster,
// and verifies one sequence at a time with every row split across its members.
constexpr int kSeqWarps = 16;
constexpr int kSeqGroups = 2;
constexpr int kSeqCluster = 2;
constexpr int kSeqStages = 3;
constexpr int kSeqChunkBytes = 4096;
// A draw task copies logits and q of the drawn row in 6 KB stages, two per warp in the
// warp's three 4 KB row stages: 1024 elements (2 KB of bf16 logits + 4 KB of q) or 768
// (3 KB of fp32 logits + 3 KB of q) per copy.
constexpr int kSeqDrawStageBytes = 6144;
constexpr int kSeqDrawElemsBf16 = 1024;
constexpr int kSeqDrawElemsF32 = 768;
constexpr int kSeqMaxDrawChunks = 512;    // chunk masses of one member's part of the drawn row
// Largest V the left-to-right kernel takes (its chunk-mass table in shared memory).
constexpr int64_t seq_max_v(specdec_dtype ldt) {
  return static_cast<int64_t>(ldt == SPECDEC_BF16 ? kSeqDrawElemsBf16 : kSeqDrawElemsF32) * kSeqMaxDrawChunks *
         kSeqCluster;
}

struct ChainParams {
  const void* logits;
  const float* q;
  const int32_t* drafts;
  const float* temps;    // nullptr in greedy-only mode
  const float* u;        // nullptr in greedy-only mode
  const int32_t* gammas; // per-sequence count of drafts to verify, or nullptr (all gamma)
  int B, gamma, V;
  int nseg;              // segments per row
  int seg;               // elements per segment
  int greedy_only;
  int host_inputs;       // left-to-right kernel: logits and q may sit in pinned host memory
  char* row_cache;       // left-to-right kernel, host-resident logits: a device copy of each
                        // sequence's latest row (B rows of V elements), or nullptr
  int drop_draws;        // left-to-right kernel, test hook: queued draws are never marked published
  unsigned long long queue_wait_ns;  // left-to-right kernel: bound on waits for queued work
  size_t counter_bytes;  // left-to-right kernel: the counter block at the workspace's start (cleared per call)
  int nch;               // streaming path: 4 KB chunks per logits row
  int nchd;              // streaming path: draw chunks per row
  int grid_stats, grid_draw;
  int nchm;              // single-read block verification: mass chunks per row
  int32_t* out_tokens;
  int32_t* out_J;
  float* out_p_draft;
  int32_t* out_status;
  ChainWorkspace ws;
};

// Single-read block verification: elements of a row per mass item (logits + q fit 4 KB).
constexpr int kBlockMassChunkBf16 = 640;
constexpr int kBlockMassChunkF32 = 512;
inline int block_mass_chunk(specdec_dtype ldt) {
  return ldt == SPECDEC_BF16 ? kBlockMassChunkBf16 : kBlockMassChunkF32;
}
constexpr int kBlockWarps = 16;    // warps per CTA, one CTA per SM
constexpr int kBlockStages = 3;    // 4 KB bulk-copy stages per warp
constexpr int kBlockSlotsS = 512;  // 4 KB chunk summaries of one row (double-buffered)
constexpr int kBlockSlotsM = 4096; // mass chunks of one sequence (all rows)

// Segment length in elements for a logits dtype and load path.
int chain_segment_len(specdec_dtype ldt, bool vector_path);
// Workspace layout; returns the total bytes (and fills ws when base != nullptr).
// path: 0 scalar loads, 1 vector loads, 2 streaming (bulk copies), 3 single-read block
// verification.
size_t chain_workspace_layout(int B, int g, int V, specdec_dtype ldt, int path,
                              void* base, ChainWorkspace* ws, size_t* counter_bytes, bool block = false);

// Streaming path: statistics, decision, draw, finish -- chained with programmatic
// dependent launch; the first launch follows ordinary stream order.
cudaError_t launch_chain_stream_stats(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream);
cudaError_t launch_chain_stream_decide(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream);
cudaError_t launch_chain_stream_draw(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream);
cudaError_t launch_chain_stream_finish(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream);
// Block verification on the streaming statistics and mass kernels.
cudaError_t launch_block_decide(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream);
cudaError_t launch_block_finish(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream);
// Block verification in one launch that reads every row once from HBM (each CTA walks
// whole sequences row by row); block_fused_fits says whether a shape fits its
// shared-memory tables.
cudaError_t launch_block_fused(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream);
bool block_fused_fits(int g, int V, specdec_dtype ldt);
int device_sm_count();
// Left-to-right chain verification reading rows only up to the first rejection: the kernel
// that clears its counter block, then the kernel itself, which (pdl) may start while the
// clearing kernel runs.
cudaError_t launch_chain_seq_clear(const ChainParams& P, cudaStream_t stream);
cudaError_t launch_chain_seq(const ChainParams& P, specdec_dtype ldt, cudaStream_t stream, bool pdl);

cudaError_t launch_chain_stats(const ChainParams& P, specdec_dtype ldt, bool vector_path,
                               cudaStream_t stream);
cudaError_t launch_chain_sample(const ChainParams& P, specdec_dtype ldt, bool vector_path,
                                cudaStream_t stream);

struct TreeParams {
  const void* logits;
  const float* q;        // recursive rejection: [B, N+1, V] drafting distributions per node
  const int32_t* node_tokens;
  const int32_t* parents;
  const float* temps;
  const float* u;
  int B, N, V, D;
  int32_t* out_tokens;
  int32_t* out_path;
  int32_t* out_J;
  int32_t* out_status;
  int wor;  // recursive rejection: children drawn without replacement
};

// The Medusa walk with rows split across a cluster of C CTAs: the cluster size for B
// sequences of V-entry rows (0 when no size fits: 16-byte rows needed), and its launch.
int tree_walk_cluster_size(int B, int V, specdec_dtype ldt);
cudaError_t launch_tree_walk_cluster(const TreeParams& P, specdec_dtype ldt, int C, cudaStream_t stream);
cudaError_t launch_tree_walk(const TreeParams& P, specdec_dtype ldt, bool vector_path,
                             cudaStream_t stream);
// Accepted-branch KV compaction (contiguous or paged caches).
struct KvCompactParams {
  char* base;
  int64_t row_bytes, slot_stride, seq_stride, block_stride, num_slots;
  const int32_t* block_table;  // nullptr: contiguous
  int block_size, max_blocks;
  int B, max_depth;
  const int32_t* prefix_len;
  const int32_t* path;
  const int32_t* num_accepted;
  int32_t* out_new_len;
  int32_t* out_status;
};
cudaError_t launch_kv_compact(const KvCompactParams& P, cudaStream_t stream);

// Sampled tree verification by recursive rejection at every node.
// Recursive rejection with rows split across a cluster of C CTAs: the cluster size for B
// sequences of V-entry rows (0 when no size fits: 16-byte rows needed), and its launch.
int tree_rr_cluster_size(int B, int V, specdec_dtype ldt);
cudaError_t launch_tree_rr_cluster(const TreeParams& P, specdec_dtype ldt, int C, cudaStream_t stream);
cudaError_t launch_tree_rr(const TreeParams& P, specdec_dtype ldt, bool vector_path, cudaStream_t stream);
// Gumbel-coupled verification and the drafter's shared-noise sampler (Philox noise).
struct GumbelParams {
  const void* logits;
  const int32_t* drafts;
  const float* temps;
  uint32_t key0, key1;
  int B, G, V, parts;
  int32_t* out_tokens;
  int32_t* out_J;
  int32_t* out_status;
  void* partials;  // workspace: [B, 2, parts] parts of the current wave's rows
  int* state;      // workspace: [B] 0 while the round is open (cleared per call)
};
cudaError_t launch_gumbel_verify(const GumbelParams& P, specdec_dtype ldt, bool vec, cudaStream_t stream);
int gumbel_parts(int B);
size_t gumbel_workspace_bytes(int B);  // [B] state (cleared per call), then the wave's parts
cudaError_t launch_gumbel_noise(uint64_t seed, int B, int R, int V, float* out, cudaStream_t stream);
cudaError_t launch_gumbel_draft(const float* q, uint64_t seed, int B, int G, int V, bool vec, int32_t* out,
                                cudaStream_t stream);
cudaError_t launch_tree_mask(const int32_t* parents, int N, int prefix_len, uint8_t* mask,
                             int64_t* pos, int32_t* depth, int32_t* status, cudaStream_t stream);

}  // namespace specdec
