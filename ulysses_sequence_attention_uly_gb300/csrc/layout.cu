// layout.cu -- the Ulysses exchange on one GPU: seq-sharded <-> head-sharded.
//
// An all-to-all is a pure permutation (sglang PR #43521, "First-sight
// check": its bytes do not depend on the transport), so with all P virtual
// ranks in one HBM the exchange is a gather of contiguous runs.  For
// seq->heads (flashdreams cp.py ContextParallelAttention._impl_ulysses;
// sglang layer.py USPAttention._forward_with_replicated_*) every gathered
// row of rank r is the run of heads [r*H/P, (r+1)*H/P) of one shard row:
// H/P * D * elem bytes, contiguous on both sides (2560 B for H=40, P=4, D=128
// bf16).  For heads->seq every output row is assembled from P such runs, and
// replicated rows are sent to every shard (the head all-gather of the
// replicated output).
//
// Kernel: one warp per run, 16-byte vector loads (streaming, read once) and
// stores, several vectors in flight per lane; grid = 8 CTAs of 8 warps per
// SM, grid-stride over runs.  HBM-bound: algorithmic bytes = 2 x bytes moved.
#include <atomic>

#include "internal.cuh"
#include "tc.cuh"

namespace uly {

// Shard whose image rows hold global image row i (shards in rank order).
__device__ __forceinline__ int image_shard(const LayoutParams& p, int i) {
  int s = 0;
  while (s + 1 < p.P && i >= p.img_off[s + 1]) ++s;
  return s;
}

// Gathered row n of rank r -> (shard, row inside the shard).
__device__ __forceinline__ void gathered_source(const LayoutParams& p, int is_kv, int r, int n, int& shard,
                                                int& row) {
  const int img = p.img_off[p.P];
  const bool prefix = (p.mode == ULY_REP_PREFIX) || (p.mode == ULY_REP_KV_PREFIX && is_kv);
  if (prefix) {
    if (n < p.R) {
      shard = r;
      row = n;
    } else {
      const int i = n - p.R;
      shard = image_shard(p, i);
      row = p.R + (i - p.img_off[shard]);
    }
  } else if (p.mode == ULY_REP_SUFFIX && n >= img) {
    shard = r;
    row = (p.img_off[r + 1] - p.img_off[r]) + (n - img);
  } else {
    shard = image_shard(p, n);
    row = n - p.img_off[shard];
  }
}

// Output row `row` of shard p -> gathered row it comes back from.
__device__ __forceinline__ int gathered_row_of_output(const LayoutParams& p, int shard, int row) {
  const int len = p.img_off[shard + 1] - p.img_off[shard];
  if (p.mode == ULY_REP_PREFIX) return row < p.R ? row : p.R + p.img_off[shard] + (row - p.R);
  if (p.mode == ULY_REP_SUFFIX) return row >= len ? p.img_off[p.P] + (row - len) : p.img_off[shard] + row;
  return p.img_off[shard] + row;
}

__device__ unsigned long long g_layout_violations;

uint64_t layout_violations(bool reset) {
  if (!kChecked) return 0;
  unsigned long long v = 0;
  if (cudaMemcpyFromSymbol(&v, g_layout_violations, sizeof v) != cudaSuccess) return ~0ull;
  if (reset) {
    const unsigned long long z = 0;
    if (cudaMemcpyToSymbol(g_layout_violations, &z, sizeof z) != cudaSuccess) return ~0ull;
  }
  return v;
}

// Source and destination of run `w` (global run index) of tensor slot t;
// false when the checked build's bounds checks reject it.  `left` receives
// how many runs from w on (w included) continue from it by fixed steps:
// to_heads, consecutive gathered rows of one segment (source row + 1 and
// destination row + 1); to_seq, consecutive ranks of one output row (the
// next rank's tensor at the same offset, destination + one rank's heads).
__device__ __forceinline__ bool run_ptrs(const LayoutParams& p, int t, int64_t w, const uint8_t*& src, uint8_t*& dst,
                                         int& left, int& r_out, int& shard_out, int64_t& src_off) {
  int64_t idx = w - p.rows_begin[t];
  const int64_t hb = p.head_bytes;
  // 32-bit division where the index fits (every practical shape): 64-bit
  // division by a runtime value costs several times as many instructions,
  // and short runs are bound by this arithmetic as much as by HBM
  const bool narrow = idx < (1LL << 31);
  if (!p.to_seq) {
    // idx = (r, b, n), n fastest
    const int N = p.dst_rows[t];
    int n, b, r;
    if (narrow) {
      const uint32_t i32 = static_cast<uint32_t>(idx), q = i32 / static_cast<uint32_t>(N);
      n = static_cast<int>(i32 - q * static_cast<uint32_t>(N));
      b = static_cast<int>(q % static_cast<uint32_t>(p.B));
      r = p.rank_lo + static_cast<int>(q / static_cast<uint32_t>(p.B));
    } else {
      n = static_cast<int>(idx % N);
      idx /= N;
      b = static_cast<int>(idx % p.B);
      r = p.rank_lo + static_cast<int>(idx / p.B);
    }
    int shard, row;
    gathered_source(p, p.is_kv[t], r, n, shard, row);
    const int hl = p.dst_heads[t], h0 = p.head_off[t];
    // the row from the segment tables and both head slices inside their tensors
    if (!(in_bounds(&g_layout_violations, row, 1, p.shard_rows[t][shard] - p.check_narrow) &&
          in_bounds(&g_layout_violations, static_cast<int64_t>(r * hl + h0) * hb, p.chunk[t],
                    static_cast<int64_t>(p.src_heads[t]) * hb) &&
          in_bounds(&g_layout_violations, static_cast<int64_t>(h0) * hb, p.chunk[t], static_cast<int64_t>(hl) * hb)))
      return false;
    src = p.src[t][shard] +
          ((static_cast<int64_t>(b) * p.shard_rows[t][shard] + row) * p.src_heads[t] + r * hl + h0) * hb;
    dst = p.dst[t][r] + ((static_cast<int64_t>(b) * N + n) * hl + h0) * hb;
    // end of n's segment in gathered rows: the replicated block or the shard's image rows
    const bool prefix = (p.mode == ULY_REP_PREFIX) || (p.mode == ULY_REP_KV_PREFIX && p.is_kv[t]);
    const int img = p.img_off[p.P];
    int seg_end;
    if (prefix)
      seg_end = n < p.R ? p.R : p.R + p.img_off[shard + 1];
    else if (p.mode == ULY_REP_SUFFIX && n >= img)
      seg_end = N;
    else
      seg_end = p.img_off[shard + 1];
    left = min(seg_end, N) - n;
    r_out = row;  // to_heads: the source row and shard, for the checks of the runs that follow
    shard_out = shard;
    src_off = static_cast<int64_t>(p.src_heads[t]) * hb;  // to_heads: source step
  } else {
    // idx = (shard, b, row, r), r fastest: the runs of one output row are
    // written by neighbouring warps; shards may differ in rows
    int shard = 0;
    while (shard + 1 < p.P && idx >= p.out_begin[shard + 1]) ++shard;
    idx -= p.out_begin[shard];
    const int rows = p.out_rows[shard];
    int r, row, b;
    if (narrow) {
      const uint32_t i32 = static_cast<uint32_t>(idx), q = i32 / static_cast<uint32_t>(p.rank_cnt);
      r = p.rank_lo + static_cast<int>(i32 - q * static_cast<uint32_t>(p.rank_cnt));
      row = static_cast<int>(q % static_cast<uint32_t>(rows));
      b = static_cast<int>(q / static_cast<uint32_t>(rows));
    } else {
      r = p.rank_lo + static_cast<int>(idx % p.rank_cnt);
      idx /= p.rank_cnt;
      row = static_cast<int>(idx % rows);
      b = static_cast<int>(idx / rows);
    }
    const int n = gathered_row_of_output(p, shard, row);
    const int hl = p.src_heads[0], h0 = p.head_off[0];
    if (!(in_bounds(&g_layout_violations, n, 1, p.src_rows[0] - p.check_narrow) &&
          in_bounds(&g_layout_violations, static_cast<int64_t>(h0) * hb, p.chunk[0], static_cast<int64_t>(hl) * hb) &&
          in_bounds(&g_layout_violations, static_cast<int64_t>(r * hl + h0) * hb, p.chunk[0],
                    static_cast<int64_t>(p.dst_heads[0]) * hb)))
      return false;
    src_off = ((static_cast<int64_t>(b) * p.src_rows[0] + n) * hl + h0) * hb;
    src = p.src[0][r] + src_off;
    dst = p.dst[0][shard] + ((static_cast<int64_t>(b) * rows + row) * p.dst_heads[0] + r * hl + h0) * hb;
    left = p.rank_lo + p.rank_cnt - r;
    r_out = r;
    shard_out = shard;
  }
  return true;
}

// Runs per warp of a slot whose runs have nv 16-byte vectors: runs of at
// most one vector per lane (<= 512 B, e.g. two bf16 heads of D = 128) go
// four to a warp in layout_kernel_short, which keeps four vectors per lane
// in flight and decodes one run of the four in full; longer runs one at a
// time in layout_kernel_long.  (Two-vector runs grouped in pairs measured
// slower than one per warp: the larger kernel holds fewer warps per SM.)
__host__ __device__ __forceinline__ int short_group(int nv) { return nv <= 0 || nv > 32 ? 0 : 4; }

__global__ void __launch_bounds__(256) layout_kernel_long(const __grid_constant__ LayoutParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  // runs of the long slots, in slot order (short slots count as empty)
  const bool l0 = !short_group(p.chunk[0] >> 4), l1 = !short_group(p.chunk[1] >> 4), l2 = !short_group(p.chunk[2] >> 4);
  const int64_t e1 = l0 ? p.rows_begin[1] - p.rows_begin[0] : 0;
  const int64_t e2 = e1 + (l1 ? p.rows_begin[2] - p.rows_begin[1] : 0);
  const int64_t e3 = e2 + (l2 ? p.rows_begin[3] - p.rows_begin[2] : 0);
  for (int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < e3; w += nwarps) {
    const int t = (w >= e1) + (w >= e2);
    const int64_t run = p.rows_begin[t] + (w - (t == 0 ? 0 : (t == 1 ? e1 : e2)));
    const uint8_t* src;
    uint8_t* dst;
    int left, rr, sh;
    int64_t so;
    if (!run_ptrs(p, t, run, src, dst, left, rr, sh, so)) continue;
    const int nv = p.chunk[t] >> 4;
    const int4* s4 = reinterpret_cast<const int4*>(src);
    int4* d4 = reinterpret_cast<int4*>(dst);
    for (int v0 = 0; v0 < nv; v0 += 128) {
      int4 buf[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int v = v0 + lane + 32 * k;
        if (v < nv) buf[k] = __ldcs(s4 + v);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int v = v0 + lane + 32 * k;
        if (v < nv) d4[v] = buf[k];
      }
    }
  }
}

__global__ void __launch_bounds__(256) layout_kernel_short(const __grid_constant__ LayoutParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t hb = p.head_bytes;
  // groups of the short slots, in slot order (long slots count as empty)
  const int u0 = short_group(p.chunk[0] >> 4), u1 = short_group(p.chunk[1] >> 4), u2 = short_group(p.chunk[2] >> 4);
  const int64_t e1 = u0 ? (p.rows_begin[1] - p.rows_begin[0] + u0 - 1) / u0 : 0;
  const int64_t e2 = e1 + (u1 ? (p.rows_begin[2] - p.rows_begin[1] + u1 - 1) / u1 : 0);
  const int64_t e3 = e2 + (u2 ? (p.rows_begin[3] - p.rows_begin[2] + u2 - 1) / u2 : 0);
  for (int64_t g = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; g < e3; g += nwarps) {
    const int t = (g >= e1) + (g >= e2);
    const int U = t == 0 ? u0 : (t == 1 ? u1 : u2);
    const int nv = p.chunk[t] >> 4;
    const int64_t first = p.rows_begin[t] + (g - (t == 0 ? 0 : (t == 1 ? e1 : e2))) * U;
    const int64_t end = p.rows_begin[t + 1];
    // the group's first run in full; the others by steps while they continue it
    const uint8_t* s0;
    uint8_t* d0;
    int left = 0, r0 = 0, sh0 = 0;
    int64_t so = 0;
    const bool ok0 = run_ptrs(p, t, first, s0, d0, left, r0, sh0, so);
    const int hl = p.to_seq ? p.src_heads[0] : p.dst_heads[t];
    const int64_t dstep = static_cast<int64_t>(hl) * hb;
    int4 buf[4];
    int4* dp[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      dp[u] = nullptr;
      const int64_t run = first + u;
      if (u >= U || run >= end) continue;
      const uint8_t* s;
      uint8_t* d;
      if (ok0 && u < left) {
        if (p.to_seq) {
          if (!in_bounds(&g_layout_violations, static_cast<int64_t>((r0 + u) * hl + p.head_off[0]) * hb, p.chunk[0],
                         static_cast<int64_t>(p.dst_heads[0]) * hb))
            continue;
          s = p.src[0][r0 + u] + so;
        } else {
          // r0 / sh0: the first run's source row and shard; so: the source step
          if (!in_bounds(&g_layout_violations, r0 + u, 1, p.shard_rows[t][sh0] - p.check_narrow)) continue;
          s = s0 + u * so;
        }
        d = d0 + u * dstep;
      } else {
        int l2_, r2_, s2_;
        int64_t o2_;
        if (!run_ptrs(p, t, run, s, d, l2_, r2_, s2_, o2_)) continue;
      }
      if (lane < nv) {
        dp[u] = reinterpret_cast<int4*>(d) + lane;
        buf[u] = __ldcs(reinterpret_cast<const int4*>(s) + lane);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (dp[u]) *dp[u] = buf[u];
  }
}

cudaError_t launch_layout(const LayoutParams& p, int64_t total_rows, int sm_count, cudaStream_t s) {
  if (total_rows <= 0) return cudaSuccess;
  // warps of each kernel: one per long run, one per group of short runs
  int64_t warps_long = 0, warps_short = 0;
  for (int t = 0; t < 3; ++t) {
    const int64_t runs = p.rows_begin[t + 1] - p.rows_begin[t];
    const int u = short_group(p.chunk[t] >> 4);
    if (u)
      warps_short += (runs + u - 1) / u;
    else
      warps_long += runs;
  }
  const int64_t cap = 8LL * sm_count;
  if (warps_long > 0) {
    const int64_t want = (warps_long + 7) / 8;
    layout_kernel_long<<<static_cast<int>(want < cap ? want : cap), 256, 0, s>>>(p);
    if (cudaGetLastError() != cudaSuccess) return cudaErrorLaunchFailure;
  }
  if (warps_short > 0) {
    const int64_t want = (warps_short + 7) / 8;
    layout_kernel_short<<<static_cast<int>(want < cap ? want : cap), 256, 0, s>>>(p);
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------ bulk copies --
// The whole exchange (every rank, every head of its slice) as block copies
// through shared memory.  to_heads: a block is up to rows_blk consecutive
// gathered rows of one (slot, rank, batch, run); the warp loads the rows from
// their shard, H * D * e bytes apart, with one cp.async.bulk per row (lane i,
// row i) and stores the block to the rank's head-major tensor, where it is
// contiguous, with one.  to_seq: a block is up to rows_blk consecutive output
// rows of one (shard, batch, run); every rank's slice of every row is loaded
// into its place in the row (one cp.async.bulk per row and rank) and the
// whole rows are stored with one.  Each CTA (one warp) keeps kBulkStages
// blocks in flight: no per-run index arithmetic in the copy loop and tens of
// KB of loads in flight per CTA whatever the run length.  The checked build
// copies row by row (and rank by rank) on both sides, each one checked, so
// that a refused run is neither read nor written.
struct BulkBlock {
  int t, r, b, n, rows, off;  // to_seq: r = the output shard
  const BulkSeg* sg;
};

// Block j -> (slot, rank or output shard, batch, run, rows).
__device__ __forceinline__ void bulk_decode(const BulkLayoutParams& p, int64_t j, BulkBlock& k) {
  const BulkSeg* sg;
  int ns, kb;
  if (p.to_seq) {
    k.t = 0;
    int sh = 0;
    while (sh + 1 < p.P && j >= p.oblocks_begin[sh + 1]) ++sh;
    sg = p.oseg[sh];
    ns = p.nos[sh];
    const uint32_t bpb = static_cast<uint32_t>(sg[ns].block0);  // blocks per batch of this shard
    const uint32_t l32 = static_cast<uint32_t>(j - p.oblocks_begin[sh]);
    const uint32_t bb = l32 / bpb;
    kb = static_cast<int>(l32 - bb * bpb);
    k.r = sh;
    k.b = static_cast<int>(bb);
  } else {
    k.t = (j >= p.blocks_begin[1]) + (j >= p.blocks_begin[2]);
    sg = p.seg[k.t];
    ns = p.nseg[k.t];
    const uint32_t bprb = static_cast<uint32_t>(sg[ns].block0);  // blocks per (rank, batch)
    const uint32_t l32 = static_cast<uint32_t>(j - p.blocks_begin[k.t]);  // < 2^31 (host-checked)
    const uint32_t rb = l32 / bprb;
    kb = static_cast<int>(l32 - rb * bprb);
    k.r = static_cast<int>(rb / static_cast<uint32_t>(p.B));
    k.b = static_cast<int>(rb - static_cast<uint32_t>(k.r) * static_cast<uint32_t>(p.B));
  }
  int s = 0;
  while (s + 1 < ns && kb >= sg[s + 1].block0) ++s;
  k.sg = sg + s;
  k.off = (kb - k.sg->block0) * p.rows_blk[k.t];
  k.rows = min(p.rows_blk[k.t], k.sg->len - k.off);
  k.n = k.sg->n0 + k.off;
}

// to_heads: row `i` of the block inside its source shard tensor; the checked
// build's row check (counted where `count`) refuses it with -1
__device__ __forceinline__ int bulk_src_row(const BulkLayoutParams& p, const BulkBlock& k, int i, int& sh,
                                            bool count) {
  sh = k.sg->shard < 0 ? k.r : k.sg->shard;
  const int srow = (k.sg->row0 < 0 ? p.img_len[sh] : k.sg->row0) + k.off + i;
  const int lim = p.shard_rows[k.t][sh] - p.check_narrow;
  if (kChecked && !count) return srow < lim ? srow : -1;
  return in_bounds(&g_layout_violations, srow, 1, lim) ? srow : -1;
}
__device__ __forceinline__ const uint8_t* bulk_src_ptr(const BulkLayoutParams& p, const BulkBlock& k, int sh,
                                                       int srow) {
  const int hl = p.run_bytes[k.t] / p.head_bytes;
  return p.src[k.t][sh] +
         ((static_cast<int64_t>(k.b) * p.shard_rows[k.t][sh] + srow) * p.heads[k.t] + k.r * hl) * p.head_bytes;
}

// Loads of block k into the stage at `stage` (all lanes); the stage's
// barrier expects the bytes actually loaded.
__device__ __forceinline__ void bulk_issue_loads(const BulkLayoutParams& p, const BulkBlock& k, uint32_t stage,
                                                 uint32_t bar, int lane) {
  const uint32_t rb = p.run_bytes[k.t];
  if (!p.to_seq) {
    int nvalid = 0;
    const uint8_t* src[kBulkMaxRows / 32];
#pragma unroll
    for (int q = 0; q < kBulkMaxRows / 32; ++q) {
      const int i = lane + 32 * q;
      src[q] = nullptr;
      if (i < k.rows) {
        int sh;
        const int srow = bulk_src_row(p, k, i, sh, true);
        if (srow >= 0) src[q] = bulk_src_ptr(p, k, sh, srow);
      }
      nvalid += src[q] != nullptr;
    }
    const int total = kChecked ? __reduce_add_sync(0xffffffffu, nvalid) : k.rows;
    if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(total) * rb);
    __syncwarp();
#pragma unroll
    for (int q = 0; q < kBulkMaxRows / 32; ++q)
      if (src[q]) bulk_load(stage + (lane + 32 * q) * rb, src[q], rb, bar);
  } else {
    // row i's slice of rank r from that rank's head-major output, into its
    // place in the assembled output row
    const int items = k.rows * p.P;
    int nvalid = 0;
    for (int it = lane; it < items; it += 32)
      nvalid += !kChecked || k.n + it / p.P < p.N[0] - p.check_narrow;
    const int total = __reduce_add_sync(0xffffffffu, nvalid);
    if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(total) * rb);
    __syncwarp();
    for (int it = lane; it < items; it += 32) {
      const int i = it / p.P, r = it - i * p.P;
      if (!in_bounds(&g_layout_violations, k.n + i, 1, p.N[0] - p.check_narrow)) continue;
      bulk_load(stage + i * p.out_row_bytes + r * rb,
                p.src[0][r] + (static_cast<int64_t>(k.b) * p.N[0] + k.n + i) * rb, rb, bar);
    }
  }
}

// Stores of block k from its stage (all lanes), then each lane commits its
// bulk group.
__device__ __forceinline__ void bulk_issue_stores(const BulkLayoutParams& p, const BulkBlock& k, uint32_t stage,
                                                  int lane) {
  const uint32_t rb = p.run_bytes[k.t];
  if (!p.to_seq) {
    uint8_t* const d0 = p.dst[k.t][k.r] + (static_cast<int64_t>(k.b) * p.N[k.t] + k.n) * rb;
    if (kChecked) {
      // (rows refused by the loads' check are left unwritten, uncounted here)
      for (int i = lane; i < k.rows; i += 32) {
        int sh;
        if (bulk_src_row(p, k, i, sh, false) >= 0 && in_bounds(&g_layout_violations, k.n + i, 1, p.N[k.t]))
          bulk_store(d0 + static_cast<int64_t>(i) * rb, stage + i * rb, rb);
      }
    } else if (lane == 0) {
      bulk_store(d0, stage, static_cast<uint32_t>(k.rows) * rb);
    }
  } else {
    const int sh = k.r;
    const int orow = (k.sg->row0 < 0 ? p.img_len[sh] : k.sg->row0) + k.off;  // first output row of the block
    uint8_t* const d0 = p.dst[0][sh] + (static_cast<int64_t>(k.b) * p.shard_rows[0][sh] + orow) * p.out_row_bytes;
    if (kChecked) {
      for (int it = lane; it < k.rows * p.P; it += 32) {
        const int i = it / p.P, r = it - i * p.P;
        if (k.n + i >= p.N[0] - p.check_narrow) continue;  // refused (and counted) by the load
        if (!in_bounds(&g_layout_violations, orow + i, 1, p.shard_rows[0][sh])) continue;
        bulk_store(d0 + static_cast<int64_t>(i) * p.out_row_bytes + r * rb, stage + i * p.out_row_bytes + r * rb,
                   rb);
      }
    } else if (lane == 0) {
      bulk_store(d0, stage, static_cast<uint32_t>(k.rows) * p.out_row_bytes);
    }
  }
  bulk_commit();
}

__global__ void __launch_bounds__(32, 1) layout_bulk_kernel(const __grid_constant__ BulkLayoutParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[kBulkStages];
  const int lane = threadIdx.x;
  const uint32_t base = (smem_u32(smem_raw) + 127u) & ~127u;
  if (lane == 0) {
    for (int s = 0; s < kBulkStages; ++s) mbar_init(smem_u32(&full[s]), 1);
    fence_mbar_init();
  }
  __syncwarp();
  const int64_t total = p.to_seq ? p.oblocks_begin[p.P] : p.blocks_begin[3];
  const int64_t first = blockIdx.x, stride = gridDim.x;
  const int64_t nblk = first < total ? (total - first + stride - 1) / stride : 0;
  volatile int never = 0;
  BulkBlock k;
  for (int64_t i = 0; i < nblk && i < kBulkStages - 1; ++i) {
    const int64_t j = first + i * stride;
    bulk_decode(p, j, k);
    bulk_issue_loads(p, k, base + static_cast<uint32_t>(i) * kBulkStage, smem_u32(&full[i]), lane);
  }
  int64_t i = 0;
  for (; i < nblk; ++i) {
    const int s = static_cast<int>(i % kBulkStages);
    const uint32_t bar = smem_u32(&full[s]);
    // (bounded: a wait that gives up records a timeout and ends the loop)
    if (!__all_sync(0xffffffffu, mbar_wait(bar, static_cast<uint32_t>(i / kBulkStages) & 1u,
                                           globaltimer_ns() + p.wait_ns, &never))) {
      if (lane == 0) atomicOr(p.status, kStatusTimeout);
      break;
    }
    const int64_t j = first + i * stride;
    bulk_decode(p, j, k);
    bulk_issue_stores(p, k, base + static_cast<uint32_t>(s) * kBulkStage, lane);
    const int64_t nx = i + kBulkStages - 1;
    if (nx < nblk) {
      // the stage of block nx last held block i - 1: its stores have read it
      bulk_wait_read<1>();
      __syncwarp();
      const int sx = static_cast<int>(nx % kBulkStages);
      const int64_t jx = first + nx * stride;
      bulk_decode(p, jx, k);
      bulk_issue_loads(p, k, base + static_cast<uint32_t>(sx) * kBulkStage, smem_u32(&full[sx]), lane);
    }
  }
  if (i < nblk) {
    // after a timeout: wait (briefly) for the loads still in flight
    const uint64_t dl = globaltimer_ns() + 100000000ull;
    for (int64_t q = i; q < nblk && q < i + kBulkStages - 1; ++q)
      mbar_wait(smem_u32(&full[q % kBulkStages]), static_cast<uint32_t>(q / kBulkStages) & 1u, dl, &never);
  }
  bulk_wait_all();
}

cudaError_t launch_layout_bulk(const BulkLayoutParams& p, int sm_count, cudaStream_t s) {
  const int64_t total = p.to_seq ? p.oblocks_begin[p.P] : p.blocks_begin[3];
  if (total <= 0) return cudaSuccess;
  constexpr int kSmem = kBulkStages * kBulkStage + 128;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
  if (!bit || !(configured.load(std::memory_order_relaxed) & bit)) {
    e = cudaFuncSetAttribute(layout_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_relaxed);
  }
  const int64_t cap = 2LL * sm_count;
  layout_bulk_kernel<<<static_cast<int>(total < cap ? total : cap), 32, kSmem, s>>>(p);
  return cudaGetLastError();
}

// One CTA row (blockIdx.y) per task, a grid-stride loop over its 16-byte
// words; used where the copy engine is slow (rows narrower than ~2 KB on a
// wide pitch) and a kernel reaches the host link's rate.
__global__ void __launch_bounds__(256) pitched_copy_kernel(const __grid_constant__ PitchedCopies p) {
  const PitchedCopy& t = p.t[blockIdx.y];
  const int64_t n = t.rows * t.w16;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / t.w16, c = i - r * t.w16;
    t.dst[r * t.pitch16 + c] = t.src[r * t.pitch16 + c];
  }
}

cudaError_t launch_pitched_copies(const PitchedCopies& p, int n_tasks, int sm_count, cudaStream_t s) {
  if (n_tasks <= 0) return cudaSuccess;
  if (n_tasks > kMaxCopyTasks) return cudaErrorInvalidValue;
  const int gx = (8 * sm_count + n_tasks - 1) / n_tasks;
  pitched_copy_kernel<<<dim3(gx, n_tasks), 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace uly
