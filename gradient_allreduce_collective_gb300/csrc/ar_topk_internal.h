// ar_topk_internal.h — launch interface of the Top-K sparsification kernels
// and of the sparse-to-dense scatter used by the sparse allreduce.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "ar_internal.h"

namespace gar {

// Tiles of the tile-shaped passes: each thread takes kTopkRuns runs of
// kTopkElems consecutive values; run u * kThreads + t of a tile belongs to
// thread t, so every load of a warp is contiguous.
constexpr int kTopkElems = 16;                                 // values per run
constexpr int kTopkRuns = 4;                                   // runs per thread
constexpr int kTopkBlock = kThreads * kTopkRuns * kTopkElems;  // values per tile
constexpr uint32_t kTopkMaxSlots = 8192;                       // slot cap per tile

// Per-rank workspace, in 32-bit words (a multiple of 64 words, 256 bytes):
//   [0, 2048)        histogram of the current radix pass
//   [2048, 2064)     TopkState
//   then nb words each of n_gt, n_eq, eq_before, out_off, n_s (nb = tiles)
//   then nb * kThreads * kTopkRuns words of run masks (used only when a
//   tile's slots overflow): for the kTopkElems values of a run, bit j (j < 16)
//   set if value j's key is above T, bit 16 + j if it equals T; the first
//   1024 of them also hold the speculative pass 1's second-digit histogram
//   (consumed before any mask is written), the next ones pass 3's match
//   list (topk_match_cap entries of two words; masks are written only when
//   the list is not used)
//   then per tile 2 * S words of slots: the indices, then the values, of the
//   tile's keys at or above the first digit's bin (every key that can be
//   kept), in index order; n_s[tile] of them
constexpr int kTopkHistWords = 2048;
constexpr int kTopkStateWords = 32;
// The next call's hint is T's magnitude times the factor of a margin level
// (rounded to nearest): a call whose candidates fell short of k (T dropped
// below its hint) widens the margin one level, kTopkTightenRun calls in a
// row that kept their candidates narrow it one level. A level outside the
// table (a fresh workspace) counts as kTopkHintStart.
constexpr int kTopkHintLevels = 6;
constexpr uint32_t kTopkHintStart = 2;
constexpr uint32_t kTopkTightenRun = 16;
__host__ __device__ inline float topk_hint_scale(uint32_t level) {
  switch (level) {
    case 0: return 0.99f;
    case 1: return 0.98f;
    case 2: return 0.95f;
    case 3: return 0.9f;
    case 4: return 0.8f;
    default: return 0.5f;
  }
}

// Entries of pass 3's match list: what the run masks hold past the second-
// digit histogram, at most 4096.
__host__ __device__ inline uint32_t topk_match_cap(uint64_t nb) {
  const uint64_t room = nb * 1024 > 1024 ? (nb * 1024 - 1024) / 2 : 0;
  return room < 4096 ? (uint32_t)room : 4096u;
}

inline uint64_t topk_blocks(uint64_t count) { return (count + kTopkBlock - 1) / kTopkBlock; }

// Slot capacity per tile: sixteen times the tile's share of k plus a margin,
// a multiple of 32, at most kTopkMaxSlots and at most a tile. The split pass
// keeps every key in the first digit's bin and above (under error feedback
// 6 to 15 times the share of k per tile: the values pile up just below the
// threshold); the speculative pass 1 keeps those at or above its hint.
inline uint32_t topk_slots(uint64_t count, uint64_t k) {
  if (count == 0) return 32;
  const uint64_t share = (k * kTopkBlock + count - 1) / count;
  uint64_t s = (16 * share + 1024 + 31) / 32 * 32;
  const uint64_t tile = count < (uint64_t)kTopkBlock ? (count + 31) / 32 * 32 : (uint64_t)kTopkBlock;
  if (s > tile) s = tile;
  if (s > kTopkMaxSlots) s = kTopkMaxSlots;
  return (uint32_t)s;
}

inline uint64_t topk_rank_words(uint64_t count, uint64_t k) {
  const uint64_t nb = topk_blocks(count);
  return (kTopkHistWords + kTopkStateWords + (5 + (uint64_t)kThreads * kTopkRuns) * nb +
          2ull * topk_slots(count, k) * nb + 63) / 64 * 64;
}

// Radix-select state of one rank, kept on the device between the passes. The
// key of a value is the bit pattern of its magnitude (sign bit cleared),
// which orders like the magnitude for every non-NaN binary32 value.
//   prefix/mask: the key bits fixed so far (after the last pass: the key T of
//                the k-th largest magnitude)
//   need:        how many keys equal to the prefix still have to be kept
//   gt:          keys strictly above the prefix (all kept)
//   ticket[p]:   blocks of pass p that have finished (the last one to finish
//                carries out the pass's single-block step)
//   overflow:    nonzero if some tile had more keys at or above the first
//                digit's bin than its slots hold; the later passes then read
//                the data instead
//   hint:        the key below which the next call's pass 1 keeps no
//                candidates: this call's T with its magnitude scaled by the
//                margin's factor; kept from call to call, any value is safe
//                (a wrong one only costs the split pass over the data)
//   spec_ok:     pass 1 filled the slots with every key at or above its hint,
//                at least k of them (so T is among them) and no tile's slots
//                overflowed: the split pass reads the slots only
//   spec_overflow: some tile had more candidates than its slots hold in pass 1
//   spec_count:  the candidates of pass 1, all tiles
//   t_prev:      the previous call's T (kept from call to call, like hint);
//                the speculative pass 1 also counts, by bits 19..10, the
//                keys in t_prev's first-digit bin
//   pre2:        that bin was this call's first digit and the slots serve:
//                pass 1 found the second digit too, the split pass is skipped
//   margin:      bits 0..7 the level of the hint's factor (topk_hint_scale),
//                bits 8.. the run of calls since it last changed that kept
//                their candidates in the slots; kept from call to call
//   mcount:      keys pass 3 found equal to the two-digit prefix (listed,
//                index and key, while they fit the match list)
//   counted:     pass 3's last block derived the per-tile counts and their
//                scans from the match list: the count pass is skipped
struct TopkState {
  uint32_t prefix;
  uint32_t mask;
  uint32_t need;
  uint32_t gt;
  uint32_t ticket[4];
  uint32_t overflow;
  uint32_t hint;
  uint32_t spec_ok;
  uint32_t spec_overflow;
  uint32_t spec_count;
  uint32_t t_prev;
  uint32_t pre2;
  uint32_t margin;
  uint32_t mcount;
  uint32_t counted;
  uint32_t pad[14];
};
static_assert(sizeof(TopkState) == kTopkStateWords * 4, "state size");

// Every rank's buffers for one Top-K call; rank r's workspace starts at
// ws + r * ws_words.
struct TopkArgs {
  const float* g[kMaxRanks];
  float* e[kMaxRanks];
  uint32_t* idx[kMaxRanks];
  float* val[kMaxRanks];
  uint32_t* ws;
  uint64_t ws_words;
  uint64_t count;
  uint64_t nb;
  uint32_t k;
  uint32_t slots;  // S, slot capacity per tile
  int nranks;
};

// Scatter of every rank's (index, value) pairs into its zeroed dense buffer;
// work is cut into tiles of kThreads pairs, tile_start[r] is rank r's first.
struct ScatterArgs {
  const uint32_t* idx[kMaxRanks];
  const float* val[kMaxRanks];
  float* dst[kMaxRanks];
  uint64_t nnz[kMaxRanks];
  uint32_t tile_start[kMaxRanks + 1];
  uint64_t count;  // pairs with an index >= count are dropped
  int nranks;
};

// Allreduce (SUM or AVG) of sparse vectors without dense copies: the output
// is cut into tiles of `tile` elements; starts[r * (ntiles + 1) + t] is the
// first pair of rank r whose index lies in tile t or later (rank r's pairs
// in ascending index order). Each block densifies every rank's pairs of one
// tile in shared memory (absent entries +0) and folds them in the ring order
// of chunk length L (or the recursive-halving order when `tree`).
struct SparseArgs {
  const uint32_t* idx[kMaxRanks];
  const float* val[kMaxRanks];
  float* dst[kMaxRanks];
  uint64_t nnz[kMaxRanks];
  uint32_t* starts;
  uint64_t count;
  uint64_t L;
  uint32_t tile;
  uint32_t ntiles;
  int nranks;
  int avg;
  int tree;
  int vec;  // every dst 16-byte aligned
};

// Tile length of the sparse fold for N ranks: N * tile floats of shared
// memory stay at 24 KiB (a multiple of 128 elements, 128..4096), so that
// eight blocks (plus the 1 KiB each reserves) fit the SM's 228 KiB.
inline uint32_t sparse_tile(int nranks) {
  uint32_t t = 6144u / (uint32_t)nranks / 128u * 128u;
  if (t < 128) t = 128;
  if (t > 4096) t = 4096;
  return t;
}
inline uint64_t sparse_ntiles(uint64_t count, int nranks) {
  return (count + sparse_tile(nranks) - 1) / sparse_tile(nranks);
}

// For every rank: a = g + e into e; (idx, val) = the k largest |a| in index
// order (ties: lower index first); e = a with those entries zeroed. `vec`:
// every g and e is 16-byte aligned.
cudaError_t launch_topk(const TopkArgs& a, bool vec, cudaStream_t stream);
cudaError_t launch_sparse_scatter(const ScatterArgs& a, cudaStream_t stream);
// max_nnz: the largest nnz over the ranks
cudaError_t launch_sparse_fold(const SparseArgs& a, uint64_t max_nnz, cudaStream_t stream);

}  // namespace gar
