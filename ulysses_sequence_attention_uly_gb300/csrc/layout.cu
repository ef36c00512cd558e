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
#include "internal.cuh"

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

__global__ void __launch_bounds__(256) layout_kernel(const __grid_constant__ LayoutParams p, int64_t total) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < total; w += nwarps) {
    const int t = (w >= p.rows_begin[1]) + (w >= p.rows_begin[2]);
    int64_t idx = w - p.rows_begin[t];
    const uint8_t* src;
    uint8_t* dst;
    const int64_t hb = p.head_bytes;
    if (!p.to_seq) {
      // idx = (r, b, n), n fastest
      const int N = p.dst_rows[t];
      const int n = static_cast<int>(idx % N);
      idx /= N;
      const int b = static_cast<int>(idx % p.B);
      const int r = p.rank_lo + static_cast<int>(idx / p.B);
      int shard, row;
      gathered_source(p, p.is_kv[t], r, n, shard, row);
      const int hl = p.dst_heads[t], h0 = p.head_off[t];
      // the row from the segment tables and both head slices inside their tensors
      if (!(in_bounds(&g_layout_violations, row, 1, p.shard_rows[t][shard] - p.check_narrow) &&
            in_bounds(&g_layout_violations, static_cast<int64_t>(r * hl + h0) * hb, p.chunk[t],
                      static_cast<int64_t>(p.src_heads[t]) * hb) &&
            in_bounds(&g_layout_violations, static_cast<int64_t>(h0) * hb, p.chunk[t], static_cast<int64_t>(hl) * hb)))
        continue;
      src = p.src[t][shard] +
            ((static_cast<int64_t>(b) * p.shard_rows[t][shard] + row) * p.src_heads[t] + r * hl + h0) * hb;
      dst = p.dst[t][r] + ((static_cast<int64_t>(b) * N + n) * hl + h0) * hb;
    } else {
      // idx = (shard, b, row, r), r fastest: the runs of one output row are
      // written by neighbouring warps; shards may differ in rows
      int shard = 0;
      while (shard + 1 < p.P && idx >= p.out_begin[shard + 1]) ++shard;
      idx -= p.out_begin[shard];
      const int rows = p.out_rows[shard];
      const int r = p.rank_lo + static_cast<int>(idx % p.rank_cnt);
      idx /= p.rank_cnt;
      const int row = static_cast<int>(idx % rows);
      const int b = static_cast<int>(idx / rows);
      const int n = gathered_row_of_output(p, shard, row);
      const int hl = p.src_heads[0], h0 = p.head_off[0];
      if (!(in_bounds(&g_layout_violations, n, 1, p.src_rows[0] - p.check_narrow) &&
            in_bounds(&g_layout_violations, static_cast<int64_t>(h0) * hb, p.chunk[0], static_cast<int64_t>(hl) * hb) &&
            in_bounds(&g_layout_violations, static_cast<int64_t>(r * hl + h0) * hb, p.chunk[0],
                      static_cast<int64_t>(p.dst_heads[0]) * hb)))
        continue;
      src = p.src[0][r] + ((static_cast<int64_t>(b) * p.src_rows[0] + n) * hl + h0) * hb;
      dst = p.dst[0][shard] + ((static_cast<int64_t>(b) * rows + row) * p.dst_heads[0] + r * hl + h0) * hb;
    }
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

cudaError_t launch_layout(const LayoutParams& p, int64_t total_rows, int sm_count, cudaStream_t s) {
  if (total_rows <= 0) return cudaSuccess;
  const int64_t want = (total_rows + 7) / 8;
  const int grid = static_cast<int>(want < 8LL * sm_count ? want : 8LL * sm_count);
  layout_kernel<<<grid, 256, 0, s>>>(p, total_rows);
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
