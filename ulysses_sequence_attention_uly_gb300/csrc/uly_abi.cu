// uly_abi.cu -- the C ABI (include/uly.h): argument validation, the plan
// (segment tables, tile-table scratch, cached TMA descriptors) and launches.
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include <cudaTypedefs.h>

#include "internal.cuh"

using namespace uly;

struct MapCacheEntry {
  bool valid = false;
  int fused = 0;
  const void* ptrs[3][kMaxRanks] = {};
  CUtensorMap tq[kMaxRanks], tk[kMaxRanks], tv[kMaxRanks];
};

// Chunks of the pipelined and host-buffer paths: one per rank, plus up to
// three more on the first rank and one on the last.
constexpr int kHostChunks = kMaxRanks + 4;

struct uly_plan {
  uly_desc d;
  int device;
  int sm_count;
  int64_t rq, rk, nq, nk;  // shard 0's rows (q, k/v), gathered rows (q, k/v)
  int32_t lens[kMaxRanks]; // image rows of each shard (all S_l for even shards)
  int64_t rq_p[kMaxRanks], rk_p[kMaxRanks];  // rows of each shard's q and k/v tensors
  int n_kv_tiles;
  void* scratch;
  uint4* tile_bits;
  int32_t* active;
  uint4* active_bits;
  uint4* active_inv;
  int32_t* n_active;
  // ring lists of uly_ring_attention: [B][P][n_kv_tiles] each
  int32_t* ring_active;
  uint4* ring_bits;
  uint4* ring_inv;
  int32_t* status;
  uint64_t wait_ns;
  int32_t withhold_fill;
  int32_t check_narrow;  // checked build, test hook: rows the layout's row checks leave out
  MapCacheEntry cache[2];
  int cache_next;
  // pipelined and host-buffer paths: streams (copies in, copies out, two for
  // attention) and events (start, tile table, inputs of chunk c in [2 + c],
  // attention of chunk c in [2 + kHostChunks + c], end)
  cudaStream_t hs[4];
  cudaEvent_t hev[3 + 2 * kHostChunks];
  bool hs_ready;
};

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int validate_desc(const uly_desc* d) {
  if (!d) return ULY_ERR_INVALID;
  if (d->B < 1 || d->P < 1 || d->S_l < 1 || d->R < 0 || d->Hq < 1 || d->Hkv < 1 || d->D < 1) return ULY_ERR_INVALID;
  if (d->rep_mode < ULY_REP_NONE || d->rep_mode > ULY_REP_KV_PREFIX) return ULY_ERR_INVALID;
  if ((d->rep_mode == ULY_REP_NONE) != (d->R == 0)) return ULY_ERR_INVALID;  // one replicated mode per call
  if (d->Hq % d->P || d->Hkv % d->P || d->Hq % d->Hkv) return ULY_ERR_INVALID;  // heads divisible by ranks
  if (d->dtype != ULY_BF16 && d->dtype != ULY_E4M3) return ULY_ERR_INVALID;
  if (d->masked_rows != ULY_ROWS_SDPA && d->masked_rows != ULY_ROWS_ZERO && d->masked_rows != ULY_ROWS_SELF)
    return ULY_ERR_INVALID;
  if (d->P > kMaxRanks) return ULY_ERR_UNSUPPORTED;
  if (d->dtype == ULY_BF16 && d->D != 64 && d->D != 128) return ULY_ERR_UNSUPPORTED;
  if (d->dtype == ULY_E4M3 && d->D != 128) return ULY_ERR_UNSUPPORTED;
  if (d->Hq > 65535 || d->B > 65535) return ULY_ERR_UNSUPPORTED;
  // row indices stay in int32 and tile indices in 20 bits
  const int64_t rows = static_cast<int64_t>(d->P) * d->S_l + d->R;
  if (rows > (1LL << 27)) return ULY_ERR_UNSUPPORTED;
  return ULY_OK;
}

int elem_size(const uly_desc& d) { return d.dtype == ULY_E4M3 ? 1 : 2; }

// Per-shard and gathered row counts from the shard lengths.
void init_rows(uly_plan* pl) {
  const uly_desc& d = pl->d;
  const bool rep_q = d.rep_mode == ULY_REP_PREFIX || d.rep_mode == ULY_REP_SUFFIX;
  const bool rep_k = d.rep_mode != ULY_REP_NONE;
  int64_t img = 0;
  for (int i = 0; i < d.P; ++i) {
    pl->rq_p[i] = pl->lens[i] + (rep_q ? d.R : 0);
    pl->rk_p[i] = pl->lens[i] + (rep_k ? d.R : 0);
    img += pl->lens[i];
  }
  pl->rq = pl->rq_p[0];
  pl->rk = pl->rk_p[0];
  pl->nq = img + (rep_q ? d.R : 0);
  pl->nk = img + (rep_k ? d.R : 0);
}

// Runs of rows in global order for q (is_kv = 0) or k/v (is_kv = 1).
int build_segs(const uly_plan* pl, int fused, int is_kv, Seg* segs) {
  const uly_desc& d = pl->d;
  const int P = d.P, R = d.R;
  const bool rep_first = d.rep_mode == ULY_REP_PREFIX || (d.rep_mode == ULY_REP_KV_PREFIX && is_kv);
  const bool rep_last = d.rep_mode == ULY_REP_SUFFIX;
  int n = 0;
  auto add = [&](int src, int row0, int len, int out_row0, int out_shard) {
    Seg s;
    s.src = src;
    s.row0 = row0;
    s.len = len;
    s.first = 0;
    s.out_row0 = out_row0;
    s.out_shard = out_shard;
    s.kv_seg = -1;
    s.pad = 0;
    segs[n++] = s;
  };
  if (rep_first) add(-1, 0, R, 0, -1);
  int off = 0;  // image rows of the shards before p
  for (int p = 0; p < P; ++p) {
    const int S = pl->lens[p];
    if (fused) {
      const int row0 = rep_first ? R : 0;
      add(p, row0, S, row0, p);
    } else {
      const int row0 = (rep_first ? R : 0) + off;
      add(-1, row0, S, row0, -1);
    }
    off += S;
  }
  // suffix rows: in the fused path they sit after each shard's own image
  // rows; `src = -1` reads the owning rank's shard, whose image length is
  // then the row offset (the kernel takes it from the segment of that rank)
  if (rep_last) add(-1, fused ? -1 : off, R, fused ? -1 : off, -1);
  // first unit (q: 256 rows) or tile (kv: 128 rows) of each run
  int acc = 0;
  const int per = is_kv ? kTileRows : kUnitRows;
  for (int i = 0; i < n; ++i) {
    segs[i].first = acc;
    acc += (segs[i].len + per - 1) / per;
  }
  if (!is_kv) {
    // kv run with the same tokens (for zero-filled masked query rows)
    const int shift = (d.rep_mode == ULY_REP_KV_PREFIX) ? 1 : 0;
    for (int i = 0; i < n; ++i) segs[i].kv_seg = i + shift;
  }
  return n;
}

int count_units(const Seg* segs, int n, int per) {
  int acc = 0;
  for (int i = 0; i < n; ++i) acc += (segs[i].len + per - 1) / per;
  return acc;
}

int encode_map(CUtensorMap* m, const void* base, int D, int heads, int64_t rows, int B, bool fp8) {
  auto enc = encode_fn();
  if (!enc) return ULY_ERR_CUDA;
  const int es = fp8 ? 1 : 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * es, static_cast<cuuint64_t>(heads) * D * es,
                           static_cast<cuuint64_t>(rows) * heads * D * es};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / es), 1, static_cast<cuuint32_t>(kTileRows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  // L2 fetch granularity: one head row of a tile (D elements) is 128 or 256
  // bytes and the next head's row follows it, so a 256-byte promotion of a
  // 128-byte row would pull another head's bytes into L2 with it
  const CUtensorMapL2promotion promo =
      D * es <= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  CUresult r = enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ULY_OK : ULY_ERR_CUDA;
}

// Plan calls run on the plan's device, which must be the current one.
int check_device(const uly_plan* pl) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return ULY_ERR_CUDA;
  return dev == pl->device ? ULY_OK : ULY_ERR_INVALID;
}

int check_ptrs(const void* const* a, int n) {
  if (!a) return ULY_ERR_INVALID;
  for (int i = 0; i < n; ++i)
    if (!a[i] || !aligned16(a[i])) return ULY_ERR_INVALID;
  return ULY_OK;
}

// Fill p.tq/tk/tv for the given tensors (cached on the pointer set).
int get_maps(uly_plan* pl, int fused, const void* const* q, const void* const* k, const void* const* v,
             AttnParams& p) {
  const uly_desc& d = pl->d;
  const int P = d.P;
  for (int c = 0; c < 2; ++c) {
    MapCacheEntry& e = pl->cache[c];
    if (!e.valid || e.fused != fused) continue;
    bool same = true;
    for (int i = 0; i < P && same; ++i)
      same = e.ptrs[0][i] == q[i] && e.ptrs[1][i] == k[i] && e.ptrs[2][i] == v[i];
    if (same) {
      memcpy(p.tq, e.tq, sizeof(p.tq));
      memcpy(p.tk, e.tk, sizeof(p.tk));
      memcpy(p.tv, e.tv, sizeof(p.tv));
      return ULY_OK;
    }
  }
  MapCacheEntry& e = pl->cache[pl->cache_next];
  pl->cache_next ^= 1;
  e.valid = false;
  const bool fp8 = d.dtype == ULY_E4M3;
  for (int i = 0; i < P; ++i) {
    int rc;
    if (fused) {
      if ((rc = encode_map(&e.tq[i], q[i], d.D, d.Hq, pl->rq_p[i], d.B, fp8))) return rc;
      if ((rc = encode_map(&e.tk[i], k[i], d.D, d.Hkv, pl->rk_p[i], d.B, fp8))) return rc;
      if ((rc = encode_map(&e.tv[i], v[i], d.D, d.Hkv, pl->rk_p[i], d.B, fp8))) return rc;
    } else {
      if ((rc = encode_map(&e.tq[i], q[i], d.D, d.Hq / P, pl->nq, d.B, fp8))) return rc;
      if ((rc = encode_map(&e.tk[i], k[i], d.D, d.Hkv / P, pl->nk, d.B, fp8))) return rc;
      if ((rc = encode_map(&e.tv[i], v[i], d.D, d.Hkv / P, pl->nk, d.B, fp8))) return rc;
    }
    e.ptrs[0][i] = q[i];
    e.ptrs[1][i] = k[i];
    e.ptrs[2][i] = v[i];
  }
  e.fused = fused;
  e.valid = true;
  memcpy(p.tq, e.tq, sizeof(p.tq));
  memcpy(p.tk, e.tk, sizeof(p.tk));
  memcpy(p.tv, e.tv, sizeof(p.tv));
  return ULY_OK;
}

// Validate an attention call and fill the launch parameters (thread-local
// storage, returned through p / tp); *groups receives the head-group count.
int setup_attention(uly_plan* pl, int fused, const void* const* q, const void* const* k, const void* const* v,
                    const uint8_t* key_mask, const int32_t* key_ranges, int32_t n_ranges, float scale,
                    int32_t head_groups, const float* q_scale, const float* k_scale, const float* v_scale,
                    void* const* o, float* const* lse, AttnParams*& pp, TileParams*& tpp, int* groups) {
  if (!pl) return ULY_ERR_INVALID;
  const uly_desc& d = pl->d;
  const int P = d.P;
  int rc;
  if ((rc = check_device(pl))) return rc;
  if ((rc = check_ptrs(q, P)) || (rc = check_ptrs(k, P)) || (rc = check_ptrs(v, P)) ||
      (rc = check_ptrs(const_cast<const void* const*>(o), P)))
    return rc;
  if (key_mask && key_ranges) return ULY_ERR_INVALID;
  if (key_ranges && n_ranges < 1) return ULY_ERR_INVALID;
  if (!(scale > 0.f) || !(scale < 3.0e38f)) return ULY_ERR_INVALID;
  const bool fp8 = d.dtype == ULY_E4M3;
  if (fp8 != (q_scale != nullptr) || fp8 != (k_scale != nullptr) || fp8 != (v_scale != nullptr))
    return ULY_ERR_INVALID;
  const int hq_l = d.Hq / P, hkv_l = d.Hkv / P;
  int g = head_groups;
  if (g == 0) g = uly_pick_head_groups(hq_l, hkv_l, pl->nq, static_cast<int64_t>(d.B) * P, pl->sm_count);
  if (g < 1 || hq_l % g || hkv_l % g) return ULY_ERR_INVALID;

  static thread_local AttnParams p;  // ~7 KB: keep it off the stack
  memset(&p, 0, sizeof(p));
  if ((rc = get_maps(pl, fused, q, k, v, p))) return rc;
  p.n_qseg = build_segs(pl, fused, 0, p.qseg);
  p.n_kseg = build_segs(pl, fused, 1, p.kseg);
  p.n_units = count_units(p.qseg, p.n_qseg, kUnitRows);
  p.n_kv_tiles = count_units(p.kseg, p.n_kseg, kTileRows);
  if (p.n_kv_tiles != pl->n_kv_tiles) return ULY_ERR_INVALID;
  for (int i = 0; i < P; ++i) p.out[i] = static_cast<uint8_t*>(o[i]);
  if (lse) {
    for (int i = 0; i < P; ++i) {
      if (!lse[i] || (reinterpret_cast<uintptr_t>(lse[i]) & 3u)) return ULY_ERR_INVALID;
      p.lse[i] = lse[i];
    }
    p.lse_out = 1;
    p.lse_row_stride = fused ? d.Hq : hq_l;
    for (int i = 0; i < P; ++i) p.lse_batch_stride[i] = (fused ? pl->rq_p[i] : pl->nq) * p.lse_row_stride;
  }
  for (int i = 0; i < P; ++i) p.shard_len[i] = pl->lens[i];
  p.fused = fused;
  p.P = P;
  p.B = d.B;
  p.Hq = d.Hq;
  p.Hkv = d.Hkv;
  p.Hq_l = hq_l;
  p.Hkv_l = hkv_l;
  p.G = d.Hq / d.Hkv;
  if (fused) {
    p.out_row_stride = static_cast<int64_t>(d.Hq) * d.D * 2;
    for (int i = 0; i < P; ++i) p.out_batch_stride[i] = pl->rq_p[i] * p.out_row_stride;
  } else {
    p.out_row_stride = static_cast<int64_t>(hq_l) * d.D * 2;
    for (int i = 0; i < P; ++i) p.out_batch_stride[i] = pl->nq * p.out_row_stride;
  }
  p.scale_log2 = scale * 1.4426950408889634f;
  p.q_scale = q_scale;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.tile_bits = pl->tile_bits;
  p.active = pl->active;
  p.active_bits = pl->active_bits;
  p.active_inv = pl->active_inv;
  p.n_active = pl->n_active;
  p.masked_rows = d.masked_rows;
  p.status = pl->status;
  p.wait_ns = pl->wait_ns;
  p.withhold_fill = pl->withhold_fill;

  static thread_local TileParams tp;
  memset(&tp, 0, sizeof(tp));
  memcpy(tp.kseg, p.kseg, sizeof(tp.kseg));
  tp.n_kseg = p.n_kseg;
  tp.n_kv_tiles = p.n_kv_tiles;
  tp.B = d.B;
  tp.Nk = static_cast<int32_t>(pl->nk);
  tp.key_mask = key_mask;
  tp.key_ranges = key_ranges;
  tp.n_ranges = key_ranges ? n_ranges : 0;
  tp.all_tiles = d.masked_rows == ULY_ROWS_SELF;
  tp.tile_bits = pl->tile_bits;
  tp.active = pl->active;
  tp.active_bits = pl->active_bits;
  tp.active_inv = pl->active_inv;
  tp.n_active = pl->n_active;
  p.group_heads = hq_l / g;
  p.group_base = 0;
  p.rank_base = 0;
  p.rank_count = P;
  pp = &p;
  tpp = &tp;
  *groups = g;
  return ULY_OK;
}

int run_attention(uly_plan* pl, int fused, const void* const* q, const void* const* k, const void* const* v,
                  const uint8_t* key_mask, const int32_t* key_ranges, int32_t n_ranges, float scale,
                  int32_t head_groups, const float* q_scale, const float* k_scale, const float* v_scale,
                  void* const* o, float* const* lse, void* stream, int merge = 0) {
  AttnParams* p;
  TileParams* tp;
  int g, rc;
  if (merge && (fused || !lse)) return ULY_ERR_INVALID;
  if ((rc = setup_attention(pl, fused, q, k, v, key_mask, key_ranges, n_ranges, scale, head_groups, q_scale,
                            k_scale, v_scale, o, lse, p, tp, &g)))
    return rc;
  p->merge = merge;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_tiles(*tp, s) != cudaSuccess) return ULY_ERR_CUDA;
  // one launch over the g head groups, processed group-major
  dim3 grid(p->n_units, pl->d.P * (pl->d.Hq / pl->d.P), pl->d.B);
  if (launch_attention(*p, pl->d.D, pl->d.dtype == ULY_E4M3, grid, s) != cudaSuccess) return ULY_ERR_CUDA;
  return ULY_OK;
}

// Chunks of the pipelined and host-buffer paths: every rank's q heads,
// except that the first rank starts with chunks of 1, 2 and 4 head groups
// (each chunk's input then arrives while the one before it attends: moving
// a head takes less than half as long as attending it) and the last head
// group of the last rank is a chunk of its own, so that little exchange is
// exposed before the first attention launch and after the last while the
// other launches stay large.  Returns the number of chunks (at most
// kHostChunks).
int make_chunks(int P, int hq_l, int g, int* ch_r, int* ch_h0, int* ch_nh) {
  const int gh = hq_l / g;
  int nc = 0;
  auto add = [&](int r, int h0, int h1) {
    if (h1 <= h0) return;
    ch_r[nc] = r;
    ch_h0[nc] = h0;
    ch_nh[nc] = h1 - h0;
    ++nc;
  };
  for (int r = 0; r < P; ++r) {
    int h = 0;
    const int end = (r == P - 1 && g > 1) ? hq_l - gh : hq_l;  // last group of the last rank apart
    if (r == 0 && g > 1) {
      for (int k = 0, n = 1; k < 3 && h + n * gh < end; ++k, n *= 2) {
        add(r, h, h + n * gh);
        h += n * gh;
      }
    }
    add(r, h, end);
    add(r, end, hq_l);
  }
  return nc;
}

// The whole exchange (every rank and head) as block copies through shared
// memory (layout_bulk_kernel): the runs of each tensor slot in gathered row
// order (the replicated rows and each shard's image rows), cut into blocks
// of up to rows_blk rows.  Returns false (nothing launched) when a run is
// wider than one block's buffer; the caller then uses the row gathers.
bool bulk_layout_params(const uly_plan* pl, int to_seq, const void* const* const* src, void* const* const* dst,
                        BulkLayoutParams& bp) {
  const uly_desc& d = pl->d;
  const int P = d.P;
  memset(&bp, 0, sizeof(bp));
  bp.P = P;
  bp.B = d.B;
  bp.to_seq = to_seq;
  bp.check_narrow = pl->check_narrow;
  bp.status = pl->status;
  bp.wait_ns = pl->wait_ns;
  for (int i = 0; i < P; ++i) bp.img_len[i] = pl->lens[i];
  const int es = to_seq ? 2 : elem_size(d);
  bp.head_bytes = d.D * es;
  if (to_seq) {
    // whole output rows of each shard: its replicated rows (prefix or suffix)
    // and its image rows, each run with the gathered row it starts from
    if (!src[0]) return false;
    bp.heads[0] = d.Hq;
    bp.run_bytes[0] = (d.Hq / P) * d.D * 2;
    bp.out_row_bytes = d.Hq * d.D * 2;
    if (bp.out_row_bytes > kBulkStage) return false;
    bp.rows_blk[0] = kBulkStage / bp.out_row_bytes < kBulkMaxRows ? kBulkStage / bp.out_row_bytes : kBulkMaxRows;
    bp.N[0] = static_cast<int32_t>(pl->nq);
    const bool rep = d.rep_mode == ULY_REP_PREFIX || d.rep_mode == ULY_REP_SUFFIX;
    const bool prefix = rep && d.rep_mode == ULY_REP_PREFIX;
    int64_t img_off = 0, total = 0;
    for (int sh = 0; sh < P; ++sh) {
      bp.src[0][sh] = static_cast<const uint8_t*>(src[0][sh]);
      bp.dst[0][sh] = static_cast<uint8_t*>(dst[0][sh]);
      bp.shard_rows[0][sh] = static_cast<int32_t>(pl->rq_p[sh]);
      int ns = 0, blocks = 0;
      auto add = [&](int len, int row0, int64_t n0) {
        if (len <= 0) return;
        BulkSeg& g = bp.oseg[sh][ns++];
        g.n0 = static_cast<int32_t>(n0);
        g.len = len;
        g.shard = sh;
        g.row0 = row0;
        g.block0 = blocks;
        blocks += (len + bp.rows_blk[0] - 1) / bp.rows_blk[0];
      };
      if (prefix) add(d.R, 0, 0);
      add(pl->lens[sh], prefix ? d.R : 0, (prefix ? d.R : 0) + img_off);
      if (rep && !prefix) add(d.R, pl->lens[sh], pl->nq - d.R);
      bp.nos[sh] = ns;
      bp.oseg[sh][ns].block0 = blocks;
      bp.oblocks_begin[sh] = total;
      total += static_cast<int64_t>(d.B) * blocks;
      img_off += pl->lens[sh];
    }
    bp.oblocks_begin[P] = total;
    return total < (1LL << 31);
  }
  int64_t total = 0;
  for (int t = 0; t < 3; ++t) {
    bp.blocks_begin[t] = total;
    if (!src[t]) continue;
    const int is_kv = t > 0;
    const int H = is_kv ? d.Hkv : d.Hq;
    bp.heads[t] = H;
    bp.run_bytes[t] = (H / P) * d.D * es;
    if (bp.run_bytes[t] > kBulkStage) return false;
    bp.rows_blk[t] = kBulkStage / bp.run_bytes[t] < kBulkMaxRows ? kBulkStage / bp.run_bytes[t] : kBulkMaxRows;
    bp.N[t] = static_cast<int32_t>(is_kv ? pl->nk : pl->nq);
    for (int i = 0; i < P; ++i) {
      bp.src[t][i] = static_cast<const uint8_t*>(src[t][i]);
      bp.dst[t][i] = static_cast<uint8_t*>(dst[t][i]);
      bp.shard_rows[t][i] = static_cast<int32_t>(is_kv ? pl->rk_p[i] : pl->rq_p[i]);
    }
    // runs in gathered row order: [replicated prefix] shard 0 .. shard P-1 [replicated suffix]
    const bool has_rep = is_kv ? d.rep_mode != ULY_REP_NONE
                               : (d.rep_mode == ULY_REP_PREFIX || d.rep_mode == ULY_REP_SUFFIX);
    const bool prefix = has_rep && d.rep_mode != ULY_REP_SUFFIX;
    const bool suffix = has_rep && d.rep_mode == ULY_REP_SUFFIX;
    int ns = 0, blocks = 0, n = 0;
    auto add = [&](int len, int shard, int row0) {
      if (len <= 0) return;
      BulkSeg& g = bp.seg[t][ns++];
      g.n0 = n;
      g.len = len;
      g.shard = shard;
      g.row0 = row0;
      g.block0 = blocks;
      blocks += (len + bp.rows_blk[t] - 1) / bp.rows_blk[t];
      n += len;
    };
    if (prefix) add(d.R, -1, 0);
    for (int i = 0; i < P; ++i) add(pl->lens[i], i, prefix ? d.R : 0);
    if (suffix) add(d.R, -1, -1);
    bp.nseg[t] = ns;
    bp.seg[t][ns].block0 = blocks;  // sentinel: blocks per (rank, batch)
    const int64_t slot_blocks = static_cast<int64_t>(P) * d.B * blocks;
    if (slot_blocks >= (1LL << 31)) return false;
    total += slot_blocks;
  }
  bp.blocks_begin[3] = total;
  return true;
}

// The exchange (to_heads, or to_seq of the output) for the ranks
// [rank_lo, rank_lo + rank_cnt) and, inside each rank's head slice, the q
// heads [h0, h0 + nh) (k/v heads [h0 / G, (h0 + nh) / G)); rank_cnt = 0
// means every rank and head (block copies where the runs fit a block).
// Chunks of ranks and heads (the pipelined path, whose exchange runs beside
// the attention kernel and must fit on its SMs) use the row gathers.
int run_layout(const uly_plan* pl, int to_seq, const void* const* const* src, void* const* const* dst,
               void* stream, int rank_lo = 0, int rank_cnt = 0, int h0 = 0, int nh = 0) {
  if (!pl) return ULY_ERR_INVALID;
  if (int rc = check_device(pl)) return rc;
  const uly_desc& d = pl->d;
  const int P = d.P;
  const int G = d.Hq / d.Hkv;
  if (rank_cnt == 0) {
    for (int t = 0; t < (to_seq ? 1 : 3); ++t) {
      if (!src[t]) continue;
      int rc;
      if ((rc = check_ptrs(src[t], P)) || (rc = check_ptrs(const_cast<const void* const*>(dst[t]), P))) return rc;
    }
    static thread_local BulkLayoutParams bp;
    if (bulk_layout_params(pl, to_seq, src, dst, bp)) {
      if (launch_layout_bulk(bp, pl->sm_count, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ULY_ERR_CUDA;
      return ULY_OK;
    }
    rank_lo = 0;
    rank_cnt = P;
    h0 = 0;
    nh = d.Hq / P;
  }
  static thread_local LayoutParams lp;
  memset(&lp, 0, sizeof(lp));
  lp.P = P;
  lp.B = d.B;
  lp.R = d.R;
  lp.rank_lo = rank_lo;
  lp.rank_cnt = rank_cnt;
  lp.check_narrow = pl->check_narrow;
  lp.img_off[0] = 0;
  for (int i = 0; i < P; ++i) lp.img_off[i + 1] = lp.img_off[i] + pl->lens[i];
  lp.mode = d.rep_mode;
  lp.to_seq = to_seq;
  const int es_in = elem_size(d);
  int64_t total = 0;
  const int nt = to_seq ? 1 : 3;
  for (int t = 0; t < 3; ++t) {
    lp.rows_begin[t] = total;
    if (t >= nt || !src[t]) continue;
    int rc;
    if ((rc = check_ptrs(src[t], P)) || (rc = check_ptrs(const_cast<const void* const*>(dst[t]), P))) return rc;
    const int is_kv = t > 0;
    const int H = is_kv ? d.Hkv : d.Hq;
    const int es = to_seq ? 2 : es_in;
    lp.head_bytes = d.D * es;
    lp.is_kv[t] = is_kv;
    for (int i = 0; i < P; ++i) {
      lp.src[t][i] = static_cast<const uint8_t*>(src[t][i]);
      lp.dst[t][i] = static_cast<uint8_t*>(dst[t][i]);
    }
    lp.head_off[t] = is_kv ? h0 / G : h0;
    lp.chunk[t] = (is_kv ? nh / G : nh) * d.D * es;
    if (!to_seq) {
      for (int i = 0; i < P; ++i) lp.shard_rows[t][i] = static_cast<int32_t>(is_kv ? pl->rk_p[i] : pl->rq_p[i]);
      lp.dst_rows[t] = static_cast<int32_t>(is_kv ? pl->nk : pl->nq);
      lp.src_heads[t] = H;
      lp.dst_heads[t] = H / P;
      total += static_cast<int64_t>(rank_cnt) * d.B * lp.dst_rows[t];
    } else {
      lp.src_rows[t] = static_cast<int32_t>(pl->nq);
      lp.src_heads[t] = H / P;
      lp.dst_heads[t] = H;
      lp.out_begin[0] = 0;
      for (int i = 0; i < P; ++i) {
        lp.out_rows[i] = static_cast<int32_t>(pl->rq_p[i]);
        lp.out_begin[i + 1] = lp.out_begin[i] + static_cast<int64_t>(d.B) * pl->rq_p[i] * rank_cnt;
      }
      total += lp.out_begin[P];
    }
  }
  lp.rows_begin[3] = total;
  for (int t = nt; t < 3; ++t) lp.rows_begin[t] = total;
  // slots skipped by a NULL source keep rows_begin[t] == rows_begin[t + 1]
  if (launch_layout(lp, total, pl->sm_count, static_cast<cudaStream_t>(stream)) != cudaSuccess) return ULY_ERR_CUDA;
  return ULY_OK;
}

}  // namespace

extern "C" {

static int plan_create(const uly_desc* desc, const int32_t* shard_lens, int device, uly_plan** out) {
  if (!out) return ULY_ERR_INVALID;
  *out = nullptr;
  if (!desc) return ULY_ERR_INVALID;
  uly_desc checked = *desc;
  if (shard_lens) checked.S_l = 1;  // ignored for uneven shards; their total is checked below
  int rc = validate_desc(&checked);
  if (rc) return rc;
  if (shard_lens) {
    int64_t img = 0;
    for (int i = 0; i < desc->P; ++i) {
      if (shard_lens[i] < 1) return ULY_ERR_INVALID;
      img += shard_lens[i];
    }
    if (img + desc->R > (1LL << 27)) return ULY_ERR_UNSUPPORTED;
  }
  uly_plan* pl = new (std::nothrow) uly_plan();
  if (!pl) return ULY_ERR_CUDA;
  pl->d = *desc;
  pl->device = device;
  pl->wait_ns = 4000000000ull;
  pl->withhold_fill = -1;
  if (cudaDeviceGetAttribute(&pl->sm_count, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
    delete pl;
    return ULY_ERR_CUDA;
  }
  const uly_desc& d = *desc;
  for (int i = 0; i < d.P; ++i) pl->lens[i] = shard_lens ? shard_lens[i] : d.S_l;
  init_rows(pl);
  Seg segs[kMaxSegs];
  const int nk = build_segs(pl, 0, 1, segs);
  pl->n_kv_tiles = count_units(segs, nk, kTileRows);
  const size_t nt = static_cast<size_t>(d.B) * pl->n_kv_tiles;
  const size_t ntr = nt * d.P;  // ring lists: one per batch and rank
  const size_t tables = (256 + nt * 16 * 3 + nt * 4 + static_cast<size_t>(d.B) * 4 + 15) / 16 * 16;
  const size_t bytes = tables + ntr * 16 * 2 + ntr * 4;
  int prev = 0;
  cudaGetDevice(&prev);
  if (cudaSetDevice(device) != cudaSuccess || cudaMalloc(&pl->scratch, bytes) != cudaSuccess) {
    cudaSetDevice(prev);
    delete pl;
    return ULY_ERR_CUDA;
  }
  cudaMemset(pl->scratch, 0, bytes);
  cudaSetDevice(prev);
  uint8_t* base = static_cast<uint8_t*>(pl->scratch);
  pl->status = reinterpret_cast<int32_t*>(base);
  pl->tile_bits = reinterpret_cast<uint4*>(base + 256);
  pl->active_bits = reinterpret_cast<uint4*>(base + 256 + nt * 16);
  pl->active_inv = reinterpret_cast<uint4*>(base + 256 + nt * 32);
  pl->active = reinterpret_cast<int32_t*>(base + 256 + nt * 48);
  pl->n_active = reinterpret_cast<int32_t*>(base + 256 + nt * 52);
  pl->ring_bits = reinterpret_cast<uint4*>(base + tables);
  pl->ring_inv = reinterpret_cast<uint4*>(base + tables + ntr * 16);
  pl->ring_active = reinterpret_cast<int32_t*>(base + tables + ntr * 32);
  *out = pl;
  return ULY_OK;
}

int uly_plan_create(const uly_desc* desc, int device, uly_plan** out) {
  return plan_create(desc, nullptr, device, out);
}

int uly_plan_create_varlen(const uly_desc* desc, const int32_t* shard_rows, int device, uly_plan** out) {
  if (!shard_rows) return ULY_ERR_INVALID;
  return plan_create(desc, shard_rows, device, out);
}

int64_t uly_plan_shard_rows(const uly_plan* plan, int32_t shard, int32_t is_kv) {
  if (!plan || shard < 0 || shard >= plan->d.P) return -1;
  return is_kv ? plan->rk_p[shard] : plan->rq_p[shard];
}

void uly_plan_destroy(uly_plan* plan) {
  if (!plan) return;
  if (plan->hs_ready) {
    for (int i = 0; i < 4; ++i) cudaStreamDestroy(plan->hs[i]);
    for (int i = 0; i < 3 + 2 * kHostChunks; ++i) cudaEventDestroy(plan->hev[i]);
  }
  if (plan->scratch) cudaFree(plan->scratch);
  delete plan;
}

int uly_plan_set_wait_limit(uly_plan* plan, uint64_t ns) {
  if (!plan || ns == 0) return ULY_ERR_INVALID;
  plan->wait_ns = ns;
  return ULY_OK;
}

int uly_plan_test_check_narrow(uly_plan* plan, int32_t rows) {
  if (!plan || rows < 0) return ULY_ERR_INVALID;
  if (!kChecked) return ULY_ERR_UNSUPPORTED;
  plan->check_narrow = rows;
  return ULY_OK;
}

int64_t uly_checked_violations(int32_t reset) {
  if (!kChecked) return -1;
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  const uint64_t a = layout_violations(reset != 0), b = attn_violations(reset != 0);
  if (a == ~0ull || b == ~0ull) return -1;
  return static_cast<int64_t>(a + b);
}

int uly_plan_test_withhold_fill(uly_plan* plan, int32_t fill) {
  if (!plan || fill < -1) return ULY_ERR_INVALID;
  plan->withhold_fill = fill;
  return ULY_OK;
}

int64_t uly_plan_rows(const uly_plan* plan, int which) {
  if (!plan) return -1;
  switch (which) {
    case 0: return plan->rq;
    case 1: return plan->rk;
    case 2: return plan->nq;
    case 3: return plan->nk;
  }
  return -1;
}

int uly_pick_head_groups(int32_t hq_local, int32_t hkv_local, int64_t q_rows, int64_t batch_ranks,
                         int32_t sm_count) {
  if (hq_local < 1 || hkv_local < 1 || q_rows < 1 || batch_ranks < 1 || sm_count < 1) return -1;
  static const int kCandidates[5] = {7, 5, 4, 3, 2};
  const int64_t tiles = (q_rows + kTileRows - 1) / kTileRows;
  for (int c : kCandidates) {
    if (hq_local % c || hkv_local % c) continue;
    if (batch_ranks * (hq_local / c) * tiles >= 4LL * sm_count) return c;
  }
  return 1;
}

int uly_to_heads(const uly_plan* plan, const void* const* q, const void* const* k, const void* const* v,
                 void* const* qh, void* const* kh, void* const* vh, void* stream) {
  if (!plan) return ULY_ERR_INVALID;
  if ((q && !qh) || (k && !kh) || (v && !vh)) return ULY_ERR_INVALID;
  const void* const* src[3] = {q, k, v};
  void* const* dst[3] = {qh, kh, vh};
  return run_layout(plan, 0, src, dst, stream);
}

int uly_to_seq(const uly_plan* plan, const void* const* oh, void* const* o, void* stream) {
  if (!plan || !oh || !o) return ULY_ERR_INVALID;
  const void* const* src[3] = {oh, nullptr, nullptr};
  void* const* dst[3] = {o, nullptr, nullptr};
  return run_layout(plan, 1, src, dst, stream);
}

int uly_attention(uly_plan* plan, const void* const* qh, const void* const* kh, const void* const* vh,
                  const uint8_t* key_mask, const int32_t* key_ranges, int32_t n_ranges, float scale,
                  int32_t head_groups, const float* q_scale, const float* k_scale, const float* v_scale,
                  void* const* oh, float* const* lse, void* stream) {
  return run_attention(plan, 0, qh, kh, vh, key_mask, key_ranges, n_ranges, scale, head_groups, q_scale, k_scale,
                       v_scale, oh, lse, stream);
}

int uly_attention_merge(uly_plan* plan, const void* const* qh, const void* const* kh, const void* const* vh,
                        const uint8_t* key_mask, const int32_t* key_ranges, int32_t n_ranges, float scale,
                        int32_t head_groups, const float* q_scale, const float* k_scale, const float* v_scale,
                        void* const* oh, float* const* lse, void* stream) {
  return run_attention(plan, 0, qh, kh, vh, key_mask, key_ranges, n_ranges, scale, head_groups, q_scale, k_scale,
                       v_scale, oh, lse, stream, 1);
}

int uly_ring_attention(uly_plan* plan, const void* const* qh, const void* const* kh, const void* const* vh,
                       const uint8_t* key_mask, const int32_t* key_ranges, int32_t n_ranges,
                       const int32_t* chunk_bounds, float scale, int32_t head_groups, const float* q_scale,
                       const float* k_scale, const float* v_scale, void* const* oh, float* const* lse,
                       void* stream) {
  if (!plan || !chunk_bounds) return ULY_ERR_INVALID;
  const int P = plan->d.P;
  if (chunk_bounds[0] != 0 || chunk_bounds[P] != plan->nk) return ULY_ERR_INVALID;
  for (int c = 0; c < P; ++c)
    if (chunk_bounds[c + 1] < chunk_bounds[c]) return ULY_ERR_INVALID;
  AttnParams* p;
  TileParams* tp;
  int g, rc;
  if ((rc = setup_attention(plan, 0, qh, kh, vh, key_mask, key_ranges, n_ranges, scale, head_groups, q_scale,
                            k_scale, v_scale, oh, lse, p, tp, &g)))
    return rc;
  // the tile table also writes each rank's rotated list; the attention
  // reads those
  tp->ring_P = P;
  for (int c = 0; c <= P; ++c) tp->ring_bounds[c] = chunk_bounds[c];
  tp->ring_active = plan->ring_active;
  tp->ring_bits = plan->ring_bits;
  tp->ring_inv = plan->ring_inv;
  p->active = plan->ring_active;
  p->active_bits = plan->ring_bits;
  p->active_inv = plan->ring_inv;
  p->ring = 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_tiles(*tp, s) != cudaSuccess) return ULY_ERR_CUDA;
  dim3 grid(p->n_units, P * (plan->d.Hq / P), plan->d.B);
  if (launch_attention(*p, plan->d.D, plan->d.dtype == ULY_E4M3, grid, s) != cudaSuccess) return ULY_ERR_CUDA;
  return ULY_OK;
}

int uly_sp_attention(uly_plan* plan, const void* const* q, const void* const* k, const void* const* v,
                     const uint8_t* key_mask, const int32_t* key_ranges, int32_t n_ranges, float scale,
                     int32_t head_groups, const float* q_scale, const float* k_scale, const float* v_scale,
                     void* const* o, float* const* lse, void* stream) {
  return run_attention(plan, 1, q, k, v, key_mask, key_ranges, n_ranges, scale, head_groups, q_scale, k_scale,
                       v_scale, o, lse, stream);
}

static int host_streams(uly_plan* pl);

int uly_pipelined_attention(uly_plan* plan, const void* const* q, const void* const* k, const void* const* v,
                            void* const* qh, void* const* kh, void* const* vh, void* const* oh,
                            const uint8_t* key_mask, const int32_t* key_ranges, int32_t n_ranges, float scale,
                            int32_t head_groups, const float* q_scale, const float* k_scale, const float* v_scale,
                            void* const* o, void* stream, void* copy_stream) {
  if (!plan || !copy_stream || stream == copy_stream) return ULY_ERR_INVALID;
  const uly_desc& d = plan->d;
  const int P = d.P;
  int rc;
  if ((rc = check_ptrs(q, P)) || (rc = check_ptrs(k, P)) || (rc = check_ptrs(v, P)) ||
      (rc = check_ptrs(const_cast<const void* const*>(qh), P)) ||
      (rc = check_ptrs(const_cast<const void* const*>(kh), P)) ||
      (rc = check_ptrs(const_cast<const void* const*>(vh), P)) ||
      (rc = check_ptrs(const_cast<const void* const*>(o), P)))
    return rc;
  AttnParams* p;
  TileParams* tp;
  int g;
  if ((rc = setup_attention(plan, 0, const_cast<const void* const*>(qh), const_cast<const void* const*>(kh),
                            const_cast<const void* const*>(vh), key_mask, key_ranges, n_ranges, scale, head_groups,
                            q_scale, k_scale, v_scale, oh, nullptr, p, tp, &g)))
    return rc;
  if ((rc = host_streams(plan))) return rc;
  const int hq_l = d.Hq / P, gh = hq_l / g;
  cudaStream_t s = static_cast<cudaStream_t>(stream), cs = static_cast<cudaStream_t>(copy_stream);
  // chunk attention alternates between two streams of the plan, so that one
  // chunk's last wave overlaps the next chunk's first
  cudaStream_t cmp[2] = {plan->hs[2], plan->hs[3]};
  cudaEvent_t* ev = plan->hev;
  // the side stream and both attention streams start after everything
  // already queued on `stream`; the second attention stream also after the
  // tile table
  if (cudaEventRecord(ev[0], s) != cudaSuccess || cudaStreamWaitEvent(cs, ev[0], 0) != cudaSuccess ||
      cudaStreamWaitEvent(cmp[0], ev[0], 0) != cudaSuccess)
    return ULY_ERR_CUDA;
  if (launch_tiles(*tp, cmp[0]) != cudaSuccess || cudaEventRecord(ev[1], cmp[0]) != cudaSuccess ||
      cudaStreamWaitEvent(cmp[1], ev[1], 0) != cudaSuccess)
    return ULY_ERR_CUDA;
  int ch_r[kHostChunks], ch_h0[kHostChunks], ch_nh[kHostChunks];
  const int nc = make_chunks(P, hq_l, g, ch_r, ch_h0, ch_nh);
  // every chunk's seq -> heads exchange, back to back on the side stream
  // (gather kernels of a few hundred microseconds in all; their CTAs fit on
  // the SMs beside the attention CTAs)
  const void* const* in_src[3] = {q, k, v};
  void* const* in_dst[3] = {qh, kh, vh};
  for (int c = 0; c < nc; ++c) {
    if ((rc = run_layout(plan, 0, in_src, in_dst, cs, ch_r[c], 1, ch_h0[c], ch_nh[c]))) return rc;
    if (cudaEventRecord(ev[2 + c], cs) != cudaSuccess) return ULY_ERR_CUDA;
  }
  // chunk c attends as soon as its inputs are in place
  for (int c = 0; c < nc; ++c) {
    cudaStream_t cc = cmp[c & 1];
    if (cudaStreamWaitEvent(cc, ev[2 + c], 0) != cudaSuccess) return ULY_ERR_CUDA;
    p->rank_base = ch_r[c];
    p->rank_count = 1;
    p->group_base = ch_h0[c] / gh;
    dim3 grid(p->n_units, ch_nh[c], d.B);
    if (launch_attention(*p, d.D, d.dtype == ULY_E4M3, grid, cc) != cudaSuccess ||
        cudaEventRecord(ev[2 + kHostChunks + c], cc) != cudaSuccess)
      return ULY_ERR_CUDA;
  }
  // finished chunks' output goes back while later chunks attend
  const void* const* out_src[3] = {const_cast<const void* const*>(oh), nullptr, nullptr};
  void* const* out_dst[3] = {o, nullptr, nullptr};
  for (int c = 0; c < nc; ++c) {
    if (cudaStreamWaitEvent(cs, ev[2 + kHostChunks + c], 0) != cudaSuccess) return ULY_ERR_CUDA;
    if ((rc = run_layout(plan, 1, out_src, out_dst, cs, ch_r[c], 1, ch_h0[c], ch_nh[c]))) return rc;
  }
  if (cudaEventRecord(ev[2 + 2 * kHostChunks], cs) != cudaSuccess ||
      cudaStreamWaitEvent(s, ev[2 + 2 * kHostChunks], 0) != cudaSuccess)
    return ULY_ERR_CUDA;
  return ULY_OK;
}

// Streams and events of the pipelined and host-buffer paths, created on
// first use on the plan's device.
static int host_streams(uly_plan* pl) {
  if (pl->hs_ready) return ULY_OK;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(pl->device) != cudaSuccess) return ULY_ERR_CUDA;
  int rc = ULY_OK;
  int ns = 0, ne = 0;
  for (; ns < 4 && rc == ULY_OK; ++ns)
    if (cudaStreamCreateWithFlags(&pl->hs[ns], cudaStreamNonBlocking) != cudaSuccess) rc = ULY_ERR_CUDA;
  for (; ne < 3 + 2 * kHostChunks && rc == ULY_OK; ++ne)
    if (cudaEventCreateWithFlags(&pl->hev[ne], cudaEventDisableTiming) != cudaSuccess) rc = ULY_ERR_CUDA;
  if (rc != ULY_OK) {
    // the failed create left nothing behind: release the ones before it
    for (int i = 0; i + 1 < ns; ++i) cudaStreamDestroy(pl->hs[i]);
    for (int i = 0; i + 1 < ne; ++i) cudaEventDestroy(pl->hev[i]);
  } else {
    pl->hs_ready = true;
  }
  cudaSetDevice(prev);
  return rc;
}

// Head slice [h0, h0 + nh) of every row of a [B, rows, H, D] tensor between
// host and device as one pitched copy.
static int copy_heads(void* dst, const void* src, int64_t rows, int H, int h0, int nh, int D, int es,
                      cudaMemcpyKind kind, cudaStream_t s) {
  const size_t pitch = static_cast<size_t>(H) * D * es, off = static_cast<size_t>(h0) * D * es;
  if (rows <= 0) return ULY_OK;
  return cudaMemcpy2DAsync(static_cast<uint8_t*>(dst) + off, pitch, static_cast<const uint8_t*>(src) + off, pitch,
                           static_cast<size_t>(nh) * D * es, static_cast<size_t>(rows), kind, s) == cudaSuccess
             ? ULY_OK
             : ULY_ERR_CUDA;
}

static int enqueue_host(uly_plan* plan, const void* const* q_host, const void* const* k_host,
                        const void* const* v_host, void* const* q, void* const* k, void* const* v,
                        const uint8_t* key_mask, const int32_t* key_ranges, int32_t n_ranges, float scale,
                        int32_t head_groups, const float* q_scale, const float* k_scale, const float* v_scale,
                        void* const* o, void* const* o_host, cudaStream_t s, bool* started);

// The device's view of a host pointer when it lies in page-locked memory
// mapped into the device's address space (every cudaHostAlloc allocation on
// a 64-bit system); null for pageable or unknown memory.  The query runs in
// relaxed capture mode, so that it is allowed while a stream is captured.
static const void* mapped_host(const void* p) {
  cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
  cudaThreadExchangeStreamCaptureMode(&mode);
  cudaPointerAttributes a;
  const bool ok = cudaPointerGetAttributes(&a, p) == cudaSuccess;
  cudaThreadExchangeStreamCaptureMode(&mode);
  if (!ok) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// Adds the head slice [h0, h0 + nh) of every row of a [B, rows, H, D]
// tensor as one pitched-copy task; false when an address, the row width or
// the pitch is not a multiple of 16 bytes (the copy engine then moves it).
static bool add_copy_task(PitchedCopies& pc, int& n, const void* src, void* dst, int64_t rows, int H, int h0,
                          int nh, int D, int es) {
  const int64_t pitch = static_cast<int64_t>(H) * D * es, off = static_cast<int64_t>(h0) * D * es;
  const int64_t width = static_cast<int64_t>(nh) * D * es;
  const uintptr_t a = reinterpret_cast<uintptr_t>(src) + off, b = reinterpret_cast<uintptr_t>(dst) + off;
  if (((a | b) & 15u) || (pitch & 15) || (width & 15) || n >= kMaxCopyTasks) return false;
  if (rows <= 0 || width == 0) return true;
  pc.t[n++] = PitchedCopy{reinterpret_cast<const int4*>(a), reinterpret_cast<int4*>(b), rows, pitch / 16,
                          static_cast<int32_t>(width / 16), 0};
  return true;
}

int uly_sp_attention_host(uly_plan* plan, const void* const* q_host, const void* const* k_host,
                          const void* const* v_host, void* const* q, void* const* k, void* const* v,
                          const uint8_t* key_mask, const int32_t* key_ranges, int32_t n_ranges, float scale,
                          int32_t head_groups, const float* q_scale, const float* k_scale, const float* v_scale,
                          void* const* o, void* const* o_host, void* stream) {
  bool started = false;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int rc = enqueue_host(plan, q_host, k_host, v_host, q, k, v, key_mask, key_ranges, n_ranges, scale,
                              head_groups, q_scale, k_scale, v_scale, o, o_host, s, &started);
  if (rc != ULY_OK && started) {
    // an enqueue failed half way: `stream` still waits for what was queued
    cudaEvent_t e = plan->hev[2 + 2 * kHostChunks];
    for (int i = 0; i < 4; ++i)
      if (cudaEventRecord(e, plan->hs[i]) == cudaSuccess) cudaStreamWaitEvent(s, e, 0);
  }
  return rc;
}

static int enqueue_host(uly_plan* plan, const void* const* q_host, const void* const* k_host,
                        const void* const* v_host, void* const* q, void* const* k, void* const* v,
                        const uint8_t* key_mask, const int32_t* key_ranges, int32_t n_ranges, float scale,
                        int32_t head_groups, const float* q_scale, const float* k_scale, const float* v_scale,
                        void* const* o, void* const* o_host, cudaStream_t s, bool* started) {
  if (!plan) return ULY_ERR_INVALID;
  const uly_desc& d = plan->d;
  const int P = d.P;
  const void* const* hosts[4] = {q_host, k_host, v_host, const_cast<const void* const*>(o_host)};
  for (int t = 0; t < 4; ++t) {
    if (!hosts[t]) return ULY_ERR_INVALID;
    for (int i = 0; i < P; ++i)
      if (!hosts[t][i]) return ULY_ERR_INVALID;
  }
  AttnParams* p;
  TileParams* tp;
  int g, rc;
  if ((rc = setup_attention(plan, 1, const_cast<const void* const*>(q), const_cast<const void* const*>(k),
                            const_cast<const void* const*>(v), key_mask, key_ranges, n_ranges, scale, head_groups,
                            q_scale, k_scale, v_scale, o, nullptr, p, tp, &g)))
    return rc;
  if ((rc = host_streams(plan))) return rc;
  const int es = elem_size(d), hq_l = d.Hq / P, hkv_l = d.Hkv / P;
  cudaStream_t h2d = plan->hs[0], d2h = plan->hs[1], cmp[2] = {plan->hs[2], plan->hs[3]};
  cudaEvent_t* ev = plan->hev;
  cudaEvent_t ev_start = ev[0], ev_tiles = ev[1], ev_end = ev[2 + 2 * kHostChunks];
  // everything starts after the work already queued on `stream`
  if (cudaEventRecord(ev_start, s) != cudaSuccess) return ULY_ERR_CUDA;
  *started = true;
  for (int i = 0; i < 4; ++i)
    if (cudaStreamWaitEvent(plan->hs[i], ev_start, 0) != cudaSuccess) return ULY_ERR_CUDA;
  if (launch_tiles(*tp, cmp[0]) != cudaSuccess || cudaEventRecord(ev_tiles, cmp[0]) != cudaSuccess ||
      cudaStreamWaitEvent(cmp[1], ev_tiles, 0) != cudaSuccess)
    return ULY_ERR_CUDA;
  // Chunks: every rank's heads, the first and the last rank split into their
  // head groups so that less copying is exposed before the first launch and
  // after the last one.  Chunk c: in, attention (alternating streams, so
  // that one chunk's last wave overlaps the next one's first), out.
  const int gh = hq_l / g, G = d.Hq / d.Hkv;
  int ch_r[kHostChunks], ch_h0[kHostChunks], ch_nh[kHostChunks];
  const int nc = make_chunks(P, hq_l, g, ch_r, ch_h0, ch_nh);
  for (int c = 0; c < nc; ++c) {
    const int r = ch_r[c], h0 = ch_h0[c], nh = ch_nh[c];
    cudaEvent_t ev_in = ev[2 + c], ev_out = ev[2 + kHostChunks + c];
    // The first chunk's copy in is exposed (no attention runs yet) and its
    // rows are narrow: with mapped page-locked shards a kernel reads them at
    // the host link's rate, where the copy engine reaches about half of it.
    bool sm_copied = false;
    if (c == 0) {
      PitchedCopies pc;
      int n = 0;
      bool can = true;
      for (int i = 0; i < P && can; ++i) {
        const int64_t rq = static_cast<int64_t>(d.B) * plan->rq_p[i], rk = static_cast<int64_t>(d.B) * plan->rk_p[i];
        const void *mq = mapped_host(q_host[i]), *mk = mapped_host(k_host[i]), *mv = mapped_host(v_host[i]);
        can = mq && mk && mv && add_copy_task(pc, n, mq, q[i], rq, d.Hq, r * hq_l + h0, nh, d.D, es) &&
              add_copy_task(pc, n, mk, k[i], rk, d.Hkv, r * hkv_l + h0 / G, nh / G, d.D, es) &&
              add_copy_task(pc, n, mv, v[i], rk, d.Hkv, r * hkv_l + h0 / G, nh / G, d.D, es);
      }
      if (can) {
        if (launch_pitched_copies(pc, n, plan->sm_count, h2d) != cudaSuccess) return ULY_ERR_CUDA;
        sm_copied = true;
      }
    }
    for (int i = 0; i < P && !sm_copied; ++i) {
      const int64_t rq = static_cast<int64_t>(d.B) * plan->rq_p[i], rk = static_cast<int64_t>(d.B) * plan->rk_p[i];
      if ((rc = copy_heads(q[i], q_host[i], rq, d.Hq, r * hq_l + h0, nh, d.D, es, cudaMemcpyHostToDevice, h2d)) ||
          (rc = copy_heads(k[i], k_host[i], rk, d.Hkv, r * hkv_l + h0 / G, nh / G, d.D, es, cudaMemcpyHostToDevice,
                           h2d)) ||
          (rc = copy_heads(v[i], v_host[i], rk, d.Hkv, r * hkv_l + h0 / G, nh / G, d.D, es, cudaMemcpyHostToDevice,
                           h2d)))
        return rc;
    }
    if (cudaEventRecord(ev_in, h2d) != cudaSuccess || cudaStreamWaitEvent(cmp[c & 1], ev_in, 0) != cudaSuccess)
      return ULY_ERR_CUDA;
    p->rank_base = r;
    p->rank_count = 1;
    p->group_base = h0 / gh;
    dim3 grid(p->n_units, nh, d.B);
    if (launch_attention(*p, d.D, d.dtype == ULY_E4M3, grid, cmp[c & 1]) != cudaSuccess ||
        cudaEventRecord(ev_out, cmp[c & 1]) != cudaSuccess || cudaStreamWaitEvent(d2h, ev_out, 0) != cudaSuccess)
      return ULY_ERR_CUDA;
    // likewise the last chunk's copy out, which follows every launch
    bool sm_out = false;
    if (c == nc - 1) {
      PitchedCopies pc;
      int n = 0;
      bool can = true;
      for (int i = 0; i < P && can; ++i) {
        const int64_t rq = static_cast<int64_t>(d.B) * plan->rq_p[i];
        void* mo = const_cast<void*>(mapped_host(o_host[i]));
        can = mo && add_copy_task(pc, n, o[i], mo, rq, d.Hq, r * hq_l + h0, nh, d.D, 2);
      }
      if (can) {
        if (launch_pitched_copies(pc, n, plan->sm_count, d2h) != cudaSuccess) return ULY_ERR_CUDA;
        sm_out = true;
      }
    }
    for (int i = 0; i < P && !sm_out; ++i) {
      const int64_t rq = static_cast<int64_t>(d.B) * plan->rq_p[i];
      if ((rc = copy_heads(o_host[i], o[i], rq, d.Hq, r * hq_l + h0, nh, d.D, 2, cudaMemcpyDeviceToHost, d2h)))
        return rc;
    }
  }
  // the last copy out follows every launch (each was waited for above)
  if (cudaEventRecord(ev_end, d2h) != cudaSuccess || cudaStreamWaitEvent(s, ev_end, 0) != cudaSuccess)
    return ULY_ERR_CUDA;
  return ULY_OK;
}

int uly_lse_merge(int64_t rows, int32_t D, const void* o_a, const float* lse_a, const void* o_b,
                  const float* lse_b, void* o_out, float* lse_out, void* stream) {
  if (rows < 0 || (D != 64 && D != 128)) return ULY_ERR_INVALID;
  if (rows == 0) return ULY_OK;
  const void* ps[6] = {o_a, lse_a, o_b, lse_b, o_out, lse_out};
  for (int i = 0; i < 6; ++i)
    if (!ps[i] || (reinterpret_cast<uintptr_t>(ps[i]) & ((i & 1) ? 3u : 15u))) return ULY_ERR_INVALID;
  int dev = 0, sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return ULY_ERR_CUDA;
  if (launch_lse_merge(rows, D, o_a, lse_a, o_b, lse_b, o_out, lse_out, sm, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return ULY_ERR_CUDA;
  return ULY_OK;
}

int uly_sync_status(uly_plan* plan, void* stream) {
  if (!plan) return ULY_ERR_INVALID;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ULY_ERR_CUDA;
  int32_t st = 0;
  if (cudaMemcpy(&st, plan->status, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess) return ULY_ERR_CUDA;
  if (st) {
    if (cudaMemset(plan->status, 0, sizeof(st)) != cudaSuccess) return ULY_ERR_CUDA;
    return ULY_ERR_TIMEOUT;
  }
  return ULY_OK;
}

const char* uly_status_string(int status) {
  switch (status) {
    case ULY_OK: return "ok";
    case ULY_ERR_INVALID: return "invalid argument";
    case ULY_ERR_UNSUPPORTED: return "unsupported configuration";
    case ULY_ERR_CUDA: return "CUDA error";
    case ULY_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

int32_t uly_device_sm_count(int device) {
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return -1;
  return n;
}

}  // extern "C"

// ------------------------------------------------------------------------
// Allocation-free fused attention (uly_sp_attention_noalloc).
//
// Some callers cannot call cudaMalloc: an application whose device memory is
// owned by its own pool (a framework's caching allocator or a serving
// runtime that reserves the GPU's memory up front) must not have a library
// allocate behind its back -- the allocation escapes the pool's accounting,
// can fail when the pool holds everything, and cudaMalloc/cudaFree
// synchronize the device.  uly_plan_create allocates its scratch with
// cudaMalloc, so those callers get this entry point instead: the same
// fused kernels, with their scratch (tile table + status word) in the
// fixed-size device array below.  Every GPU that loads the library holds
// the array until the process exits.
namespace {

constexpr int kNoAllocMaxTiles = 4096;  // B * (kv tiles of 128 keys)
constexpr size_t kNoAllocBytes = 256 + static_cast<size_t>(kNoAllocMaxTiles) * (16 + 16 + 16 + 4 + 4);

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

namespace {

// Device address of g_noalloc_scratch in the current device's context.  The
// array's name is only a host-side stand-in, so the address is looked up on
// every call: a host-side table lookup that allocates nothing, and that stays
// right when the context is torn down and created again (cudaDeviceReset),
// where an address kept from an earlier context would point at freed memory.
int noalloc_scratch(uint8_t** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return ULY_ERR_CUDA;
  *out = static_cast<uint8_t*>(p);
  return ULY_OK;
}

}  // namespace

extern "C" int uly_sp_attention_noalloc(const uly_desc* desc, const void* const* q, const void* const* k,
                                        const void* const* v, const uint8_t* key_mask, const int32_t* key_ranges,
                                        int32_t n_ranges, float scale, int32_t head_groups, const float* q_scale,
                                        const float* k_scale, const float* v_scale, void* const* o,
                                        float* const* lse, void* stream) {
  int rc = validate_desc(desc);
  if (rc) return rc;
  const uly_desc& d = *desc;
  const int P = d.P;
  if ((rc = check_ptrs(q, P)) || (rc = check_ptrs(k, P)) || (rc = check_ptrs(v, P)) ||
      (rc = check_ptrs(const_cast<const void* const*>(o), P)))
    return rc;
  if (key_mask && key_ranges) return ULY_ERR_INVALID;
  if (key_ranges && n_ranges < 1) return ULY_ERR_INVALID;
  if (!(scale > 0.f) || !(scale < 3.0e38f)) return ULY_ERR_INVALID;
  const bool fp8 = d.dtype == ULY_E4M3;
  if (fp8 != (q_scale != nullptr) || fp8 != (k_scale != nullptr) || fp8 != (v_scale != nullptr))
    return ULY_ERR_INVALID;

  // shape bookkeeping of a plan, kept in thread-local storage (no heap)
  static thread_local uly_plan pl;
  pl.d = d;
  for (int i = 0; i < P; ++i) pl.lens[i] = d.S_l;
  init_rows(&pl);
  int sm_count = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return ULY_ERR_CUDA;

  static thread_local AttnParams p;
  memset(&p, 0, sizeof(p));
  p.n_qseg = build_segs(&pl, 1, 0, p.qseg);
  p.n_kseg = build_segs(&pl, 1, 1, p.kseg);
  p.n_units = count_units(p.qseg, p.n_qseg, kUnitRows);
  p.n_kv_tiles = count_units(p.kseg, p.n_kseg, kTileRows);
  if (static_cast<int64_t>(d.B) * p.n_kv_tiles > kNoAllocMaxTiles) return ULY_ERR_UNSUPPORTED;

  const int hq_l = d.Hq / P, hkv_l = d.Hkv / P;
  int g = head_groups;
  if (g == 0) g = uly_pick_head_groups(hq_l, hkv_l, pl.nq, static_cast<int64_t>(d.B) * P, sm_count);
  if (g < 1 || hq_l % g || hkv_l % g) return ULY_ERR_INVALID;

  uint8_t* scratch = nullptr;
  if ((rc = noalloc_scratch(&scratch))) return rc;
  int32_t* status = reinterpret_cast<int32_t*>(scratch);
  uint4* tile_bits = reinterpret_cast<uint4*>(scratch + 256);
  uint4* active_bits = reinterpret_cast<uint4*>(scratch + 256 + static_cast<size_t>(kNoAllocMaxTiles) * 16);
  uint4* active_inv = reinterpret_cast<uint4*>(scratch + 256 + static_cast<size_t>(kNoAllocMaxTiles) * 32);
  int32_t* active = reinterpret_cast<int32_t*>(scratch + 256 + static_cast<size_t>(kNoAllocMaxTiles) * 48);
  int32_t* n_active = reinterpret_cast<int32_t*>(scratch + 256 + static_cast<size_t>(kNoAllocMaxTiles) * 52);

  for (int i = 0; i < P; ++i) {
    if ((rc = encode_map(&p.tq[i], q[i], d.D, d.Hq, pl.rq, d.B, fp8))) return rc;
    if ((rc = encode_map(&p.tk[i], k[i], d.D, d.Hkv, pl.rk, d.B, fp8))) return rc;
    if ((rc = encode_map(&p.tv[i], v[i], d.D, d.Hkv, pl.rk, d.B, fp8))) return rc;
    p.out[i] = static_cast<uint8_t*>(o[i]);
  }
  if (lse) {
    for (int i = 0; i < P; ++i) {
      if (!lse[i] || (reinterpret_cast<uintptr_t>(lse[i]) & 3u)) return ULY_ERR_INVALID;
      p.lse[i] = lse[i];
    }
    p.lse_out = 1;
    p.lse_row_stride = d.Hq;
    for (int i = 0; i < P; ++i) p.lse_batch_stride[i] = pl.rq * d.Hq;
  }
  for (int i = 0; i < P; ++i) p.shard_len[i] = d.S_l;
  p.fused = 1;
  p.P = P;
  p.B = d.B;
  p.Hq = d.Hq;
  p.Hkv = d.Hkv;
  p.Hq_l = hq_l;
  p.Hkv_l = hkv_l;
  p.G = d.Hq / d.Hkv;
  p.out_row_stride = static_cast<int64_t>(d.Hq) * d.D * 2;
  for (int i = 0; i < P; ++i) p.out_batch_stride[i] = pl.rq * p.out_row_stride;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.q_scale = q_scale;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.tile_bits = tile_bits;
  p.active = active;
  p.active_bits = active_bits;
  p.active_inv = active_inv;
  p.n_active = n_active;
  p.masked_rows = d.masked_rows;
  p.status = status;
  p.wait_ns = 4000000000ull;
  p.withhold_fill = -1;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the status word must start at zero; the tile table is rewritten in full
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return ULY_ERR_CUDA;
  static thread_local TileParams tp;
  memset(&tp, 0, sizeof(tp));
  memcpy(tp.kseg, p.kseg, sizeof(tp.kseg));
  tp.n_kseg = p.n_kseg;
  tp.n_kv_tiles = p.n_kv_tiles;
  tp.B = d.B;
  tp.Nk = static_cast<int32_t>(pl.nk);
  tp.key_mask = key_mask;
  tp.key_ranges = key_ranges;
  tp.n_ranges = key_ranges ? n_ranges : 0;
  tp.all_tiles = d.masked_rows == ULY_ROWS_SELF;
  tp.tile_bits = tile_bits;
  tp.active = active;
  tp.active_bits = active_bits;
  tp.active_inv = active_inv;
  tp.n_active = n_active;
  if (launch_tiles(tp, s) != cudaSuccess) return ULY_ERR_CUDA;
  // one launch over the g head groups, processed group-major
  p.group_heads = hq_l / g;
  p.rank_base = 0;
  p.rank_count = P;
  dim3 grid(p.n_units, P * hq_l, d.B);
  if (launch_attention(p, d.D, fp8, grid, s) != cudaSuccess) return ULY_ERR_CUDA;
  return ULY_OK;
}

extern "C" int uly_noalloc_sync_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ULY_ERR_CUDA;
  int32_t st = 0;
  if (cudaMemcpyFromSymbol(&st, g_noalloc_scratch, sizeof(st)) != cudaSuccess) return ULY_ERR_CUDA;
  if (st) {
    const int32_t z = 0;
    if (cudaMemcpyToSymbol(g_noalloc_scratch, &z, sizeof(z)) != cudaSuccess) return ULY_ERR_CUDA;
    return ULY_ERR_TIMEOUT;
  }
  return ULY_OK;
}
