// internal.cuh -- structures shared by the library's translation units (host
// planning code and the kernels).  Not part of the public ABI.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/uly.h"

namespace uly {

constexpr int kMaxRanks = ULY_MAX_RANKS;

// ------------------------------------------------------- checked build --
// Built with -DULY_CHECKED=1, the kernels check every index they compute
// into a global tensor (a row taken from the segment tables, a head slice)
// against that tensor's extent; an index outside it is counted in a device
// counter of its translation unit and the access is skipped, so nothing
// traps or faults.  In the normal build the checks compile to nothing.
#if defined(ULY_CHECKED) && ULY_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

// [off, off + len) inside [0, extent)?  Counts a violation in *counter when
// not (checked build); always true in the normal build.
__device__ __forceinline__ bool in_bounds(unsigned long long* counter, int64_t off, int64_t len, int64_t extent) {
  if (!kChecked) return true;
  if (off >= 0 && len >= 0 && off + len <= extent) return true;
  atomicAdd(counter, 1ull);
  return false;
}

// Violations counted since the last reset by each translation unit's
// kernels (0 in the normal build); the caller has synchronised the device.
uint64_t layout_violations(bool reset);
uint64_t attn_violations(bool reset);
constexpr int kMaxSegs = kMaxRanks + 1;  // P image runs + one replicated run
constexpr int kTileRows = 128;           // rows of one q or kv tile (tcgen05 M = 128)
constexpr int kUnitRows = 2 * kTileRows; // q rows per CTA (two softmax warpgroups)

// status word bits written by kernels (atomicOr)
constexpr int kStatusTimeout = 1;

// ---------------------------------------------------------------- layout --
// One byte-moving pass: every "row copy" moves `chunk[t]` contiguous bytes.
struct LayoutParams {
  const uint8_t* src[3][kMaxRanks];
  uint8_t* dst[3][kMaxRanks];
  int64_t rows_begin[4];  // prefix of row copies per tensor slot
  int32_t chunk[3];       // bytes per row copy, multiple of 16
  int32_t src_rows[3];    // rows of one source tensor (per batch)
  int32_t dst_rows[3];    // rows of one destination tensor (per batch)
  int32_t src_heads[3];   // heads of a source row
  int32_t dst_heads[3];   // heads of a destination row
  int32_t is_kv[3];
  int32_t head_bytes;     // D * element size
  int32_t P, B, R, mode;
  int32_t to_seq;         // 0: seq->heads, 1: heads->seq
  int32_t img_off[kMaxRanks + 1];          // image rows of the shards before shard p (prefix sums)
  int32_t shard_rows[3][kMaxRanks];        // rows of shard p's tensor (seq->heads sources)
  int32_t out_rows[kMaxRanks];             // rows of shard p's output (heads->seq destinations)
  int64_t out_begin[kMaxRanks + 1];        // heads->seq: row copies before shard p
  int32_t rank_lo, rank_cnt;               // ranks moved: [rank_lo, rank_lo + rank_cnt)
  int32_t head_off[3];                     // first head moved, inside each rank's slice
  int32_t check_narrow;                    // checked build, test hook: rows the row checks leave out
};

// The exchange as block copies through shared memory (layout_bulk_kernel):
// a run of consecutive gathered rows of one tensor slot that come from (or go
// to) consecutive rows of one shard -- the replicated rows or one shard's
// image rows.  Listed in gathered row order.
struct BulkSeg {
  int32_t n0;      // first gathered row
  int32_t len;     // rows
  int32_t shard;   // to_heads: source shard (-1: the rank's own copy of the replicated rows)
  int32_t row0;    // first row inside the shard's tensor; -1 (to_heads): right after the shard's image rows
  int32_t block0;  // first block of the run inside one (rank, batch), or (to_seq) one (shard, batch)
  int32_t pad[3];
};

struct BulkLayoutParams {
  const uint8_t* src[3][kMaxRanks];
  uint8_t* dst[3][kMaxRanks];
  // to_heads: runs of each tensor slot (+ a sentinel holding the block count
  // per (rank, batch)); to_seq: runs of output rows of each shard (+ a
  // sentinel holding the block count per batch).  One or the other, so they
  // share their storage.
  union {
    BulkSeg seg[3][kMaxSegs + 1];
    BulkSeg oseg[kMaxRanks][3];
  };
  int32_t nseg[3];
  int32_t run_bytes[3];          // one gathered row of one rank: H/P * D * e
  int32_t rows_blk[3];           // gathered rows per block
  int32_t heads[3];              // heads of a shard row (to_heads source / to_seq destination)
  int32_t N[3];                  // gathered rows of a rank's tensor
  int32_t shard_rows[3][kMaxRanks];  // rows of each shard's tensor (per batch)
  int32_t img_len[kMaxRanks];    // image rows of each shard
  int64_t blocks_begin[4];       // prefix over slots of P * B * blocks per (rank, batch)
  // to_seq: blocks are whole output rows of one shard (every rank's slice
  // gathered into shared memory, then one contiguous store): per shard its
  // number of runs (oseg above), and the prefix over shards of B * blocks
  // per batch
  int32_t nos[kMaxRanks];
  int64_t oblocks_begin[kMaxRanks + 1];
  int32_t out_row_bytes;         // Hq * D * 2
  int32_t head_bytes;            // D * e
  int32_t P, B, to_seq;
  int32_t check_narrow;          // checked build, test hook: rows the row checks leave out
  int32_t* status;               // device status word (bounded waits)
  uint64_t wait_ns;
};
constexpr int kBulkStage = 24 * 1024;  // shared-memory bytes of one block
constexpr int kBulkStages = 4;
constexpr int kBulkMaxRows = 64;

// ------------------------------------------------------------- attention --
// A run of consecutive rows of one tensor: either a shard's image rows or the
// replicated rows.  Segments are listed in global key (and query) order.
struct Seg {
  int32_t src;        // tensor map index; -1 = the rank that owns the head
  int32_t row0;       // first row of the run inside that tensor; -1 = right after the
                      // image rows of that shard (a replicated suffix of uneven shards)
  int32_t len;        // rows
  int32_t first;      // q: first 256-row unit of the run; kv: first 128-row tile
  int32_t out_row0;   // q: first output row (-1: after the image rows of each output shard)
  int32_t out_shard;  // q, fused: output shard; -1 = every shard (replicated rows)
  int32_t kv_seg;     // q: kv run holding the same tokens (-1: none)
  int32_t pad;
};

struct AttnParams {
  CUtensorMap tq[kMaxRanks];
  CUtensorMap tk[kMaxRanks];
  CUtensorMap tv[kMaxRanks];
  uint8_t* out[kMaxRanks];
  float* lse[kMaxRanks];     // optional log-sum-exp outputs (lse_out != 0)
  int64_t lse_row_stride;                     // floats
  int64_t lse_batch_stride[kMaxRanks];        // floats, per output tensor
  int32_t lse_out;
  Seg qseg[kMaxSegs];
  Seg kseg[kMaxSegs];
  int32_t n_qseg, n_kseg, n_units, n_kv_tiles;
  int32_t fused;
  int32_t P, B, Hq, Hkv, Hq_l, Hkv_l, G;
  int32_t shard_len[kMaxRanks];  // image rows of each shard
  int32_t group_heads;  // local q heads per rank in one head group (Hq_l / g)
  int32_t group_base;   // first head group of this launch (grid.y covers the following groups)
  int32_t rank_base;    // first rank of this launch
  int32_t rank_count;   // ranks covered by this launch (P for a whole call)
  int64_t out_row_stride;                     // bytes
  int64_t out_batch_stride[kMaxRanks];        // bytes, per output tensor (shards may differ in rows)
  float scale_log2;                          // softmax scale * log2(e)
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  const uint4* tile_bits;   // [B][n_kv_tiles] admitted keys of each kv tile
  const int32_t* active;    // [B][n_kv_tiles] (seg << 20 | tile) of tiles with an admitted key
  const uint4* active_bits; // [B][n_kv_tiles] tile_bits of those tiles, in the same order
  const uint4* active_inv;  // [B][n_kv_tiles] their keys that are not admitted (a masked row's key set)
  const int32_t* n_active;  // [B]
  int32_t masked_rows;      // ULY_ROWS_SDPA / ULY_ROWS_ZERO / ULY_ROWS_SELF
  int32_t* status;
  uint64_t wait_ns;
  int32_t withhold_fill;    // test hook: index of a K/V fill the loader never issues (-1 = none)
  // staged path: merge into the running (O, LSE) already in out / lse.  Kept
  // last: a field inserted earlier moves the others' offsets in the kernel's
  // parameter block, which changed the e4m3 kernel's register allocation
  // (156 -> 159) and cost it 3%.
  int32_t merge;
  // staged path, uly_ring_attention: the kv tile lists are per batch and
  // rank ([B][P][n_kv_tiles]), each rank's starting at its own key chunk
  int32_t ring;
};

struct TileParams {
  Seg kseg[kMaxSegs];
  int32_t n_kseg, n_kv_tiles, B, Nk;
  const uint8_t* key_mask;    // [B][Nk] or null
  const int32_t* key_ranges;  // [B][n_ranges][2] or null
  int32_t n_ranges;
  int32_t all_tiles;          // list every tile that has keys (masked rows attend to masked keys)
  uint4* tile_bits;
  int32_t* active;
  uint4* active_bits;
  uint4* active_inv;
  int32_t* n_active;
  // ring lists (uly_ring_attention; ring_P = 0: none): the batch's list
  // rotated for each of ring_P ranks, rank c's starting at the first tile
  // whose first key is at or after ring_bounds[c]
  int32_t ring_P;
  int32_t ring_bounds[kMaxRanks + 1];
  int32_t* ring_active;
  uint4* ring_bits;
  uint4* ring_inv;
};

// Pitched copies between host and device buffers of the same row layout,
// run by SMs (the source or destination is page-locked host memory mapped
// into the device's address space): task i copies `rows` rows of `w16`
// 16-byte words, row r at word r * pitch16 of both src and dst.
struct PitchedCopy {
  const int4* src;
  int4* dst;
  int64_t rows;
  int64_t pitch16;
  int32_t w16;
  int32_t pad;
};
constexpr int kMaxCopyTasks = 3 * kMaxRanks;
struct PitchedCopies {
  PitchedCopy t[kMaxCopyTasks];
};

// launchers (defined in the .cu files)
cudaError_t launch_layout(const LayoutParams& p, int64_t total_rows, int sm_count, cudaStream_t s);
cudaError_t launch_layout_bulk(const BulkLayoutParams& p, int sm_count, cudaStream_t s);
cudaError_t launch_pitched_copies(const PitchedCopies& p, int n_tasks, int sm_count, cudaStream_t s);
cudaError_t launch_tiles(const TileParams& p, cudaStream_t s);
cudaError_t launch_attention(const AttnParams& p, int D, bool fp8, dim3 grid, cudaStream_t s);
cudaError_t launch_lse_merge(int64_t rows, int D, const void* o_a, const float* lse_a, const void* o_b,
                             const float* lse_b, void* o_out, float* lse_out, int sm_count, cudaStream_t s);

}  // namespace uly
