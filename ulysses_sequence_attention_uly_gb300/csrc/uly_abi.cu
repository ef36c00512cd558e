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

struct uly_plan {
  uly_desc d;
  int device;
  int sm_count;
  int64_t rq, rk, nq, nk;  // shard rows (q, k/v), gathered rows (q, k/v)
  int n_kv_tiles;
  void* scratch;
  uint4* tile_bits;
  int32_t* active;
  uint4* active_bits;
  int32_t* n_active;
  int32_t* status;
  uint64_t wait_ns;
  int32_t withhold_fill;
  MapCacheEntry cache[2];
  int cache_next;
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
  if (d->masked_rows != ULY_ROWS_SDPA && d->masked_rows != ULY_ROWS_ZERO) return ULY_ERR_INVALID;
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

// Runs of rows in global order for q (is_kv = 0) or k/v (is_kv = 1).
int build_segs(const uly_plan* pl, int fused, int is_kv, Seg* segs) {
  const uly_desc& d = pl->d;
  const int P = d.P, S = d.S_l, R = d.R;
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
  for (int p = 0; p < P; ++p) {
    if (fused) {
      const int row0 = rep_first ? R : 0;
      add(p, row0, S, row0, p);
    } else {
      const int row0 = (rep_first ? R : 0) + p * S;
      add(-1, row0, S, row0, -1);
    }
  }
  if (rep_last) add(-1, fused ? S : P * S, R, fused ? S : P * S, -1);
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
  CUresult r = enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ULY_OK : ULY_ERR_CUDA;
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
      if ((rc = encode_map(&e.tq[i], q[i], d.D, d.Hq, pl->rq, d.B, fp8))) return rc;
      if ((rc = encode_map(&e.tk[i], k[i], d.D, d.Hkv, pl->rk, d.B, fp8))) return rc;
      if ((rc = encode_map(&e.tv[i], v[i], d.D, d.Hkv, pl->rk, d.B, fp8))) return rc;
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

int run_attention(uly_plan* pl, int fused, const void* const* q, const void* const* k, const void* const* v,
                  const uint8_t* key_mask, const int32_t* key_ranges, int32_t n_ranges, float scale,
                  int32_t head_groups, const float* q_scale, const float* k_scale, const float* v_scale,
                  void* const* o, float* const* lse, void* stream) {
  if (!pl) return ULY_ERR_INVALID;
  const uly_desc& d = pl->d;
  const int P = d.P;
  int rc;
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
    p.lse_batch_stride = (fused ? pl->rq : pl->nq) * p.lse_row_stride;
  }
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
    p.out_batch_stride = pl->rq * p.out_row_stride;
  } else {
    p.out_row_stride = static_cast<int64_t>(hq_l) * d.D * 2;
    p.out_batch_stride = pl->nq * p.out_row_stride;
  }
  p.scale_log2 = scale * 1.4426950408889634f;
  p.q_scale = q_scale;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.tile_bits = pl->tile_bits;
  p.active = pl->active;
  p.active_bits = pl->active_bits;
  p.n_active = pl->n_active;
  p.zero_masked_rows = d.masked_rows == ULY_ROWS_ZERO;
  p.status = pl->status;
  p.wait_ns = pl->wait_ns;
  p.withhold_fill = pl->withhold_fill;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
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
  tp.tile_bits = pl->tile_bits;
  tp.active = pl->active;
  tp.active_bits = pl->active_bits;
  tp.n_active = pl->n_active;
  if (launch_tiles(tp, s) != cudaSuccess) return ULY_ERR_CUDA;

  // one launch over the g head groups, processed group-major
  p.group_heads = hq_l / g;
  dim3 grid(p.n_units, P * hq_l, d.B);
  if (launch_attention(p, d.D, fp8, grid, s) != cudaSuccess) return ULY_ERR_CUDA;
  return ULY_OK;
}

int run_layout(const uly_plan* pl, int to_seq, const void* const* const* src, void* const* const* dst,
               void* stream) {
  if (!pl) return ULY_ERR_INVALID;
  const uly_desc& d = pl->d;
  const int P = d.P;
  static thread_local LayoutParams lp;
  memset(&lp, 0, sizeof(lp));
  lp.P = P;
  lp.B = d.B;
  lp.S_l = d.S_l;
  lp.R = d.R;
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
    lp.chunk[t] = (H / P) * d.D * es;
    if (!to_seq) {
      lp.src_rows[t] = static_cast<int32_t>(is_kv ? pl->rk : pl->rq);
      lp.dst_rows[t] = static_cast<int32_t>(is_kv ? pl->nk : pl->nq);
      lp.src_heads[t] = H;
      lp.dst_heads[t] = H / P;
      total += static_cast<int64_t>(P) * d.B * lp.dst_rows[t];
    } else {
      lp.src_rows[t] = static_cast<int32_t>(pl->nq);
      lp.dst_rows[t] = static_cast<int32_t>(pl->rq);
      lp.src_heads[t] = H / P;
      lp.dst_heads[t] = H;
      total += static_cast<int64_t>(P) * d.B * lp.dst_rows[t] * P;
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

int uly_plan_create(const uly_desc* desc, int device, uly_plan** out) {
  if (!out) return ULY_ERR_INVALID;
  *out = nullptr;
  int rc = validate_desc(desc);
  if (rc) return rc;
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
  const int64_t img = static_cast<int64_t>(d.P) * d.S_l;
  const bool has_rep = d.rep_mode != ULY_REP_NONE;
  pl->rq = (d.rep_mode == ULY_REP_PREFIX || d.rep_mode == ULY_REP_SUFFIX) ? d.S_l + d.R : d.S_l;
  pl->rk = has_rep ? d.S_l + d.R : d.S_l;
  pl->nq = (d.rep_mode == ULY_REP_PREFIX || d.rep_mode == ULY_REP_SUFFIX) ? img + d.R : img;
  pl->nk = has_rep ? img + d.R : img;
  Seg segs[kMaxSegs];
  const int nk = build_segs(pl, 0, 1, segs);
  pl->n_kv_tiles = count_units(segs, nk, kTileRows);
  const size_t nt = static_cast<size_t>(d.B) * pl->n_kv_tiles;
  const size_t bytes = 256 + nt * 16 + nt * 16 + nt * 4 + static_cast<size_t>(d.B) * 4;
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
  pl->active = reinterpret_cast<int32_t*>(base + 256 + nt * 32);
  pl->n_active = reinterpret_cast<int32_t*>(base + 256 + nt * 36);
  *out = pl;
  return ULY_OK;
}

void uly_plan_destroy(uly_plan* plan) {
  if (!plan) return;
  if (plan->scratch) cudaFree(plan->scratch);
  delete plan;
}

int uly_plan_set_wait_limit(uly_plan* plan, uint64_t ns) {
  if (!plan || ns == 0) return ULY_ERR_INVALID;
  plan->wait_ns = ns;
  return ULY_OK;
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

int uly_sp_attention(uly_plan* plan, const void* const* q, const void* const* k, const void* const* v,
                     const uint8_t* key_mask, const int32_t* key_ranges, int32_t n_ranges, float scale,
                     int32_t head_groups, const float* q_scale, const float* k_scale, const float* v_scale,
                     void* const* o, float* const* lse, void* stream) {
  return run_attention(plan, 1, q, k, v, key_mask, key_ranges, n_ranges, scale, head_groups, q_scale, k_scale,
                       v_scale, o, lse, stream);
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
constexpr size_t kNoAllocBytes = 256 + static_cast<size_t>(kNoAllocMaxTiles) * (16 + 16 + 4 + 4);
constexpr int kNoAllocMaxDevices = 64;

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

namespace {

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (the array's name is only a host-side stand-in).
int noalloc_scratch(uint8_t** out) {
  static std::mutex mu;
  static void* addr[kNoAllocMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ULY_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return ULY_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return ULY_ERR_CUDA;
    addr[dev] = p;
  }
  *out = static_cast<uint8_t*>(addr[dev]);
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
  const int64_t img = static_cast<int64_t>(P) * d.S_l;
  const bool rep_q = d.rep_mode == ULY_REP_PREFIX || d.rep_mode == ULY_REP_SUFFIX;
  pl.rq = rep_q ? d.S_l + d.R : d.S_l;
  pl.rk = d.rep_mode != ULY_REP_NONE ? d.S_l + d.R : d.S_l;
  pl.nq = rep_q ? img + d.R : img;
  pl.nk = d.rep_mode != ULY_REP_NONE ? img + d.R : img;
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
  int32_t* active = reinterpret_cast<int32_t*>(scratch + 256 + static_cast<size_t>(kNoAllocMaxTiles) * 32);
  int32_t* n_active = reinterpret_cast<int32_t*>(scratch + 256 + static_cast<size_t>(kNoAllocMaxTiles) * 36);

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
    p.lse_batch_stride = pl.rq * d.Hq;
  }
  p.fused = 1;
  p.P = P;
  p.B = d.B;
  p.Hq = d.Hq;
  p.Hkv = d.Hkv;
  p.Hq_l = hq_l;
  p.Hkv_l = hkv_l;
  p.G = d.Hq / d.Hkv;
  p.out_row_stride = static_cast<int64_t>(d.Hq) * d.D * 2;
  p.out_batch_stride = pl.rq * p.out_row_stride;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.q_scale = q_scale;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.tile_bits = tile_bits;
  p.active = active;
  p.active_bits = active_bits;
  p.n_active = n_active;
  p.zero_masked_rows = d.masked_rows == ULY_ROWS_ZERO;
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
  tp.tile_bits = tile_bits;
  tp.active = active;
  tp.active_bits = active_bits;
  tp.n_active = n_active;
  if (launch_tiles(tp, s) != cudaSuccess) return ULY_ERR_CUDA;
  // one launch over the g head groups, processed group-major
  p.group_heads = hq_l / g;
  dim3 grid(p.n_units, P * hq_l, d.B);
  if (launch_attention(p, d.D, fp8, grid, s) != cudaSuccess) return ULY_ERR_CUDA;
  return ULY_OK;
}
