// Accepted-branch KV compaction after a tree round.
//
// SD 20.5, "Keeping the caches consistent after a rejection": the verification pass wrote
// a cache entry for every candidate; after the round only the accepted branch is kept,
// and for a tree its entries sit among discarded siblings, so they are gathered into
// consecutive slots (a chain only moves its length).  Node i of sequence b sits at
// logical slot prefix[b] + i; the entry of path[b][d] moves to slot prefix[b] + d.
//
// A path climbs the tree (path[d] >= d, strictly increasing), so a move never reads a slot
// that an earlier move wrote; it may read the slot a later move writes (path [1, 2] reads
// slot 1 before filling it).  Every thread moves the same byte offsets at every depth, so
// it loads a batch of depths into registers before it stores any of them: the loads of a
// batch are in flight together, and no read can see a later move's write.  Grid: (row
// chunks, sequences); each CTA moves its byte range of the row at every depth.  Contiguous caches address slot s of sequence b at
// base + b * seq_stride + s * slot_stride; paged caches at base + block_table[b][s / bs] *
// block_stride + (s % bs) * slot_stride.

#include "specdec_device.cuh"
#include "specdec_internal.h"

namespace specdec {

namespace {

constexpr int kCompactThreads = 256;
constexpr int64_t kCompactChunk = 16 * 1024;  // bytes of a row per CTA

__global__ void __launch_bounds__(kCompactThreads) kv_compact_kernel(const KvCompactParams P, bool vec16) {
  __shared__ int s_ok;
  const int b = blockIdx.y;
  const int64_t lo = static_cast<int64_t>(blockIdx.x) * kCompactChunk;
  const int64_t hi = min(P.row_bytes, lo + kCompactChunk);
  const int J = __ldg(P.num_accepted + b);
  const int P0 = __ldg(P.prefix_len + b);
  const int32_t* path = P.path + static_cast<int64_t>(b) * P.max_depth;
  if (threadIdx.x == 0) {  // the path must climb the tree and stay inside the cache
    int ok = J >= 0 && J <= P.max_depth && P0 >= 0 ? 1 : 0;
    int prev = -1;
    for (int d = 0; ok && d < J; ++d) {
      const int s = __ldg(path + d);
      if (s < d || s <= prev || static_cast<int64_t>(P0) + s >= P.num_slots) ok = 0;
      prev = s;
    }
    if (J < 0) ok = -1;  // a failed round: nothing to move, the length stays
    s_ok = ok;
    if (blockIdx.x == 0) {
      if (P.out_new_len) P.out_new_len[b] = ok == 1 ? P0 + J : P0;
      if (P.out_status) P.out_status[b] = ok == 0 ? SPECDEC_STATUS_BAD_TREE : 0;
    }
  }
  __syncthreads();
  if (s_ok != 1) return;
  auto slot = [&](int s) -> char* {
    if (P.block_table) {
      const int blk = __ldg(P.block_table + static_cast<int64_t>(b) * P.max_blocks + s / P.block_size);
      return P.base + static_cast<int64_t>(blk) * P.block_stride + static_cast<int64_t>(s % P.block_size) * P.slot_stride;
    }
    return P.base + static_cast<int64_t>(b) * P.seq_stride + static_cast<int64_t>(s) * P.slot_stride;
  };
  constexpr int kBatch = 4;  // depths whose loads are in flight together
  for (int d0 = 0; d0 < J; d0 += kBatch) {
    const int nd = min(kBatch, J - d0);
    if (vec16) {
      constexpr int U = 4;  // 16-byte vectors per thread per depth: 256 threads x 64 B = the 16 KB chunk
      static_assert(U * 16 * kCompactThreads == kCompactChunk, "one pass covers the chunk");
      const int64_t o0 = lo + 16 * static_cast<int64_t>(threadIdx.x);
      uint4 v[kBatch][U];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        if (i < nd) {
          const int d = d0 + i, s = __ldg(path + d);
          if (s != d) {
            const char* src = slot(P0 + s);
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const int64_t oo = o0 + 16 * static_cast<int64_t>(u) * kCompactThreads;
              if (oo < hi) v[i][u] = *reinterpret_cast<const uint4*>(src + oo);
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        if (i < nd) {
          const int d = d0 + i, s = __ldg(path + d);
          if (s != d) {
            char* dst = slot(P0 + d);
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const int64_t oo = o0 + 16 * static_cast<int64_t>(u) * kCompactThreads;
              if (oo < hi) *reinterpret_cast<uint4*>(dst + oo) = v[i][u];
            }
          }
        }
      }
    } else {
      for (int64_t o = lo + threadIdx.x; o < hi; o += kCompactThreads) {
        char v[kBatch];
        for (int i = 0; i < nd; ++i) {
          const int d = d0 + i, s = __ldg(path + d);
          v[i] = s != d ? slot(P0 + s)[o] : 0;
        }
        for (int i = 0; i < nd; ++i) {
          const int d = d0 + i, s = __ldg(path + d);
          if (s != d) slot(P0 + d)[o] = v[i];
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_kv_compact(const KvCompactParams& P, cudaStream_t stream) {
  const bool vec16 = (reinterpret_cast<uintptr_t>(P.base) % 16 == 0) && P.row_bytes % 16 == 0 &&
                     P.slot_stride % 16 == 0 && (P.block_table ? P.block_stride % 16 == 0 : P.seq_stride % 16 == 0);
  const int64_t chunks = (P.row_bytes + kCompactChunk - 1) / kCompactChunk;
  return launch_kernel(kv_compact_kernel, dim3(static_cast<unsigned>(chunks), static_cast<unsigned>(P.B)),
                       dim3(kCompactThreads), 0, stream, 0, P, vec16);
}

}  // namespace specdec
