// attn.cu -- joint text+image attention for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes (sglang layer.py LocalAttention.forward and the
// attn_impl.forward calls of USPAttention): for every query row, softmax over
// the admitted keys of scale * q.k, times V; GQA maps q head h to kv head
// h / (Hq/Hkv); e4m3 inputs carry per-head scales (LightX2V PR #1235).  A
// query with no admitted key gets 0.
//
// How (one CTA = one (batch, head, 256-query-row unit)):
//   warp 8      TMA producer: the two 128-row Q tiles once, then K and V
//               tiles of every kv tile that has an admitted key, through a
//               ring of kSlots shared-memory slots (K_0, V_0, K_1, V_1, ...);
//               fills travel in pairs (V_j, K_j+1) with one full and one
//               empty barrier per pair.
//   warp 9      one thread issues tcgen05.mma from descriptor tables built
//               once per CTA:
//                 S_i = Q_i K^T        (SS, both K-major, f32 in TMEM)
//                 O_i += P_i V         (TS: P_i read from TMEM, V MN-major)
//               in the order S0(0) S1(0) | PV0(j) S0(j+1) PV1(j) S1(j+1) ...
//               so the tensor core works on one tile while the softmax
//               warpgroup of the other tile runs.
//   warps 0-3   softmax of Q tile 0, warps 4-7 of Q tile 1: one thread per
//               query row (= TMEM lane); online softmax in the log2 domain
//               with a lazily updated reference max (the running O and sum
//               are rescaled only when the max grows by more than 2^8);
//               P (bf16 or e4m3) is written back into the S columns of TMEM; the epilogue
//               divides by the row sum and stores bf16 rows.
// TMEM: S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D,256+2D).
//
// Work per (b, h, q row) does not depend on the grid, the head group or the
// path (staged or fused), so head-group splits and the fused path are
// bit-identical to one whole call.
//
// Every mbarrier wait is bounded (globaltimer deadline); a wait that gives up
// records a timeout in the status word, tells the other roles through a
// shared flag, and the CTA drains its outstanding copies and MMAs, frees TMEM
// and returns.
#include <atomic>

#include "internal.cuh"
#include "tc.cuh"

namespace uly {

template <int D, bool FP8>
struct Cfg {
  static constexpr int kElem = FP8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElem;             // bytes of one head row
  static constexpr int kPanels = kRowBytes / 128;          // 128-byte swizzle panels per row
  static constexpr int kPanelBytes = kTileRows * 128;      // 16 KB
  static constexpr int kTileBytes = kPanels * kPanelBytes; // one 128-row tile
  static constexpr int kBoxInner = 128 / kElem;            // elements of one panel row
  static constexpr int kSlots = (D == 128 && !FP8) ? 4 : 8;
  static constexpr int kQkSteps = kRowBytes / 32;          // K = 32 bytes per MMA
  static constexpr int kPvSteps = FP8 ? 4 : 8;             // 128 kv rows / (32 or 16)
  static constexpr int kPvRowsPerStep = FP8 ? 32 : 16;
  static constexpr uint32_t kFmt = FP8 ? 0u : 1u;          // e4m3 / bf16
  static constexpr uint32_t kIdescS = make_idesc(kFmt, 128, 128, 0, 0);
  static constexpr uint32_t kIdescO = make_idesc(kFmt, 128, D, 0, 1);
  // e4m3: P goes through shared memory (two buffers per Q tile, 128 rows x
  // 128 keys of one byte, K-major with the 128-byte swizzle), so that the S
  // columns of TMEM are free as soon as the softmax has read them
  static constexpr bool kPsmem = FP8;
  static constexpr int kPTileBytes = kTileRows * 128;
  static constexpr int kSmem = 1024 + 2 * kTileBytes + kSlots * kTileBytes + (kPsmem ? 4 * kPTileBytes : 0);
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kThreads = 320;
};

struct Bars {
  uint64_t q_full;
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t s_full[2];
  uint64_t s_free[2];     // e4m3: S of Q tile 0 / 1 read out of TMEM
  // P of Q tile i stored: [i][0] (TMEM P), or [i][j mod 2] for kv tile j
  // (e4m3: one barrier per shared-memory buffer, since that softmax can
  // run a kv tile ahead of the issuer's wait for the previous P)
  uint64_t p_full[2][2];
  uint64_t o_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ unsigned long long g_attn_violations;

// log-sum-exp of a row's admitted scores (natural log): sum exp(s) =
// l * 2^m_ref, since p = 2^(s * log2(e) * scale - m_ref); -inf for a row
// written as zero or with no admitted key.
__device__ __forceinline__ float row_lse(bool zero, float l_run, float m_ref) {
  return (zero || !(l_run > 0.f)) ? -INFINITY : (m_ref + lg2_approx(l_run)) * 0.6931471805599453f;
}

uint64_t attn_violations(bool reset) {
  if (!kChecked) return 0;
  unsigned long long v = 0;
  if (cudaMemcpyFromSymbol(&v, g_attn_violations, sizeof v) != cudaSuccess) return ~0ull;
  if (reset) {
    const unsigned long long z = 0;
    if (cudaMemcpyToSymbol(g_attn_violations, &z, sizeof z) != cudaSuccess) return ~0ull;
  }
  return v;
}

__device__ __forceinline__ void record_timeout(const AttnParams& p, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicOr(p.status, kStatusTimeout);
}

// Bits [base, base + 32) of "column c < n" for a 128-column tile.
__device__ __forceinline__ uint32_t lane_mask(int n, int base) {
  const int k = n - base;
  return k >= 32 ? 0xFFFFFFFFu : (k <= 0 ? 0u : ((1u << k) - 1u));
}

// Masked keys of a partial tile become -inf (their exponential is exactly 0).
__device__ __forceinline__ void mask_tile(uint32_t (&a)[4][32], const uint4 bits) {
  const uint32_t ninf = __float_as_uint(-INFINITY);
  const uint32_t w[4] = {bits.x, bits.y, bits.z, bits.w};
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int k = 0; k < 32; ++k)
      if (!((w[c] >> k) & 1u)) a[c][k] = ninf;
}

// Row max of the 128 scores: four independent chains of three-input max.
__device__ __forceinline__ float row_max(const uint32_t (&a)[4][32]) {
  float m[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    m[c] = -INFINITY;
#pragma unroll
    for (int k = 0; k < 32; k += 2) m[c] = max3f(m[c], __uint_as_float(a[c][k]), __uint_as_float(a[c][k + 1]));
  }
  return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

// p = 2^(s * sl2 + neg) for the 32-score chunks [C0, C1) of one row's 128
// scores, rounded to bf16 and written to TMEM at tP as the P operand of the
// PV MMA (column j holds kv 2j, 2j+1), one chunk at a time; returns the sum
// of the f32 values.  The exponentials run on the MUFU, whose ex2 rate on
// GB300 covers the bf16 MMAs.
template <int C0, int C1>
__device__ __forceinline__ float tile_exp_store(const uint32_t (&a)[4][32], float sl2, float neg, uint32_t tP) {
  const uint64_t mul = f2(sl2, sl2), add = f2(neg, neg);
  uint64_t acc[4] = {f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
  for (int c = C0; c < C1; ++c) {
    uint32_t pk[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      uint64_t x = f2_fma(f2(__uint_as_float(a[c][2 * q]), __uint_as_float(a[c][2 * q + 1])), mul, add);
      float x0, x1;
      f2_split(x, x0, x1);
      x = f2(ex2_approx(x0), ex2_approx(x1));
      acc[q & 3] = f2_add(acc[q & 3], x);
      float p0, p1;
      f2_split(x, p0, p1);
      pk[q] = pack_bf16x2(p0, p1);
    }
    tmem_st16(tP + 16 * c, pk);
  }
  const uint64_t t = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
  float s0, s1;
  f2_split(t, s0, s1);
  return s0 + s1;
}

// S_i = Q_i K^T for one 128-key tile from precomputed descriptors of the
// Q tile and the K slot (both K-major, 128-byte swizzle), accumulator at
// TMEM d.
template <int D, bool FP8>
__device__ __forceinline__ void issue_s(uint32_t d, const uint64_t (&dq)[Cfg<D, FP8>::kQkSteps],
                                        const uint64_t (&dk)[Cfg<D, FP8>::kQkSteps]) {
  using C = Cfg<D, FP8>;
#pragma unroll
  for (int k = 0; k < C::kQkSteps; ++k) {
    if (FP8)
      mma_f8_ss(d, dq[k], dk[k], C::kIdescS, k > 0);
    else
      mma_bf16_ss(d, dq[k], dk[k], C::kIdescS, k > 0);
  }
}

// O_i (+)= P_i V for one 128-key tile (bf16): P packed in TMEM at a, V slot
// from precomputed descriptors (MN-major), accumulator at TMEM d.
template <int D, bool FP8>
__device__ __forceinline__ void issue_pv(uint32_t d, uint32_t a, const uint64_t (&dv)[Cfg<D, FP8>::kPvSteps],
                                         bool acc) {
  using C = Cfg<D, FP8>;
  static_assert(!FP8, "e4m3 P is read from shared memory (issue_pv_ss)");
#pragma unroll
  for (int k = 0; k < C::kPvSteps; ++k) mma_bf16_ts(d, a + 8 * k, dv[k], C::kIdescO, acc || k > 0);
}

// O_i (+)= P_i V with P_i in shared memory (e4m3): both operands from
// precomputed descriptors (P K-major, V MN-major), accumulator at TMEM d.
template <int D, bool FP8>
__device__ __forceinline__ void issue_pv_ss(uint32_t d, const uint64_t (&dp)[Cfg<D, FP8>::kPvSteps],
                                            const uint64_t (&dv)[Cfg<D, FP8>::kPvSteps], bool acc) {
  using C = Cfg<D, FP8>;
#pragma unroll
  for (int k = 0; k < C::kPvSteps; ++k) mma_f8_ss(d, dp[k], dv[k], C::kIdescO, acc || k > 0);
}

// The e4m3 counterpart of tile_exp_store, for all 128 keys of the row.  P is
// rounded to e4m3 (three mantissa bits) for the PV MMA, so the exponentials
// are taken in f16, two per MUFU instruction, and converted straight to
// e4m3; the row sum adds eight pairs (values of at most 2^8) in f16x2 before
// going to f32.  With half the MUFU instructions the softmax keeps up with
// the fp8 MMAs, which run at twice the bf16 rate.  P goes to shared memory
// as the row's 128 bytes of a K-major P tile with the 128-byte swizzle
// (16-byte chunk c of row r at chunk c ^ (r mod 8); rows 128 bytes apart,
// eight-row groups 1024 bytes apart), the A operand of an SS MMA.
// row_addr = the row's first byte, r7 = r mod 8.  Returns the row sum.
__device__ __forceinline__ float tile_exp_store_e4m3_smem(const uint32_t (&a)[4][32], float sl2, float neg,
                                                          uint32_t row_addr, uint32_t r7) {
  const uint64_t mul = f2(sl2, sl2), add = f2(neg, neg);
  uint64_t acc = f2(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t pk[8];
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      uint32_t hs = 0u;
      uint16_t bt[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int q = 8 * g + t;
        float x0, x1;
        f2_split(f2_fma(f2(__uint_as_float(a[c][2 * q]), __uint_as_float(a[c][2 * q + 1])), mul, add), x0, x1);
        const uint32_t e = ex2_f16x2(pack_f16x2(x0, x1));
        hs = t == 0 ? e : add_f16x2(hs, e);
        bt[t] = e4m3x2_from_f16x2(e);
      }
#pragma unroll
      for (int t = 0; t < 4; ++t) pk[4 * g + t] = pack_b16x2(bt[2 * t], bt[2 * t + 1]);
      float s0, s1;
      f16x2_to_f32(hs, s0, s1);
      acc = f2_add(acc, f2(s0, s1));
      // keys 32c + 16g .. +15 = 16-byte chunk 2c + g of the row
      st_shared_v4(row_addr + ((static_cast<uint32_t>(2 * c + g) ^ r7) << 4), pk[4 * g], pk[4 * g + 1],
                   pk[4 * g + 2], pk[4 * g + 3]);
    }
  }
  float s0, s1;
  f2_split(acc, s0, s1);
  return s0 + s1;
}

// MERGE: the epilogue merges into the running (O, LSE) already in the
// outputs (uly_attention_merge); a separate instance, so that the plain
// kernels carry none of its code.
template <int D, bool FP8, bool MERGE>
__global__ void __launch_bounds__(320, 1) attn_kernel(const __grid_constant__ AttnParams p) {
  using C = Cfg<D, FP8>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Bars bars;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  // ---- which work unit
  const int u = blockIdx.x;
  int qs = 0;
  while (qs + 1 < p.n_qseg && u >= p.qseg[qs + 1].first) ++qs;
  const Seg qseg = p.qseg[qs];
  const int unit_row = (u - qseg.first) * kUnitRows;       // first row of the unit inside the run
  const bool two = unit_row + kTileRows < qseg.len;        // is Q tile 1 inside the run?
  // blockIdx.y walks the head groups in order (group-major): group, rank,
  // head inside the group; a group holds group_heads local heads of each of
  // the ranks [rank_base, rank_base + rank_count)
  const int per_group = p.rank_count * p.group_heads;
  const int grp = p.group_base + blockIdx.y / per_group;
  const int r = p.rank_base + (blockIdx.y % per_group) / p.group_heads;
  const int j = grp * p.group_heads + blockIdx.y % p.group_heads;  // local q head of rank r
  const int h = r * p.Hq_l + j;                                 // global q head
  const int hk = h / p.G;                                       // global kv head
  const int b = blockIdx.z;
  const int n_it = p.n_active[b];
  // kv tile list: one per batch, or (ring) one per batch and rank, each
  // rank's list starting at its own key chunk
  const int64_t list = p.ring ? static_cast<int64_t>(b) * p.P + r : b;
  const int32_t* active = p.active + list * p.n_kv_tiles;

  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = sbase;                         // two Q tiles
  const uint32_t sKV = sbase + 2 * C::kTileBytes;    // ring of kSlots tiles
  const uint32_t sP = sKV + C::kSlots * C::kTileBytes;  // e4m3: P of tile i, buffer k at 2i + k
  volatile int* abort_flag = &bars.abort_flag;

  const uint32_t b_qfull = smem_u32(&bars.q_full);
  const uint32_t b_drain = smem_u32(&bars.drain);
  if (tid == 0) {
    mbar_init(b_qfull, 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(smem_u32(&bars.full[s]), 1);
      mbar_init(smem_u32(&bars.empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars.s_full[i]), 1);
      mbar_init(smem_u32(&bars.s_free[i]), 4);
      mbar_init(smem_u32(&bars.p_full[i][0]), 4);
      mbar_init(smem_u32(&bars.p_full[i][1]), 4);
      mbar_init(smem_u32(&bars.o_done[i]), 1);
    }
    mbar_init(b_drain, 1);
    bars.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(&bars.tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  const uint64_t deadline = globaltimer_ns() + p.wait_ns;

  if (warp == 8) {
    // ================================================= TMA producer ==
    if (lane == 0) {
      const int qmap = qseg.src < 0 ? r : qseg.src;
      const CUtensorMap* mq = &p.tq[qmap];
      const int qhead = p.fused ? h : j;
      const int kvhead = p.fused ? hk : j / p.G;
      const int q_row0 = qseg.row0 < 0 ? p.shard_len[qmap] : qseg.row0;
      mbar_arrive_expect_tx(b_qfull, (two ? 2 : 1) * C::kTileBytes);
      for (int i = 0; i < (two ? 2 : 1); ++i)
        for (int pn = 0; pn < C::kPanels; ++pn)
          tma_load_4d(sQ + i * C::kTileBytes + pn * C::kPanelBytes, mq, b_qfull, pn * C::kBoxInner, qhead,
                      q_row0 + unit_row + i * kTileRows, b);
      // K/V fills go in groups that share one pair of ring slots and one
      // full / empty barrier: group 0 = K(0), group g = V(g-1) + K(g),
      // group n_it = V(n_it-1).  Group g uses slots 2g-1 and 2g (mod slots)
      // and reuses those of group g - kSlots/2 once the MMAs released it.
      constexpr int kHalf = C::kSlots / 2;
      int g = 0;
      for (; g <= n_it; ++g) {
        const int bi = g % kHalf;
        if (g >= kHalf) {
          if (!mbar_wait(smem_u32(&bars.empty[bi]), ((g / kHalf) - 1) & 1, deadline, abort_flag)) {
            record_timeout(p, abort_flag);
            break;
          }
        }
        const bool has_v = g > 0, has_k = g < n_it;
        const uint32_t bf = smem_u32(&bars.full[bi]);
        mbar_arrive_expect_tx(bf, (has_v && has_k ? 2 : 1) * C::kTileBytes);
        for (int part = 0; part < 2; ++part) {
          const bool is_v = part == 0;
          if (is_v ? !has_v : !has_k) continue;
          const int c = is_v ? 2 * g - 1 : 2 * g;  // fill index: K(j) = 2j, V(j) = 2j + 1
          if (c == p.withhold_fill) continue;
          const int slot = c % C::kSlots;
          const int e = active[c >> 1];
          if (!in_bounds(&g_attn_violations, e >> 20, 1, p.n_kseg)) continue;
          const Seg& ks = p.kseg[e >> 20];
          const int kmap = ks.src < 0 ? r : ks.src;
          const CUtensorMap* m = is_v ? &p.tv[kmap] : &p.tk[kmap];
          const int k_row0 = ks.row0 < 0 ? p.shard_len[kmap] : ks.row0;
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_load_4d(sKV + slot * C::kTileBytes + pn * C::kPanelBytes, m, bf, pn * C::kBoxInner, kvhead,
                        k_row0 + (e & 0xFFFFF) * kTileRows, b);
        }
      }
      if (*abort_flag) {
        // drain: wait (briefly) for every group still in flight so no copy
        // lands in shared memory after the CTA has left (a group with a
        // withheld fill never completes and only costs the short bound)
        const uint64_t dl2 = globaltimer_ns() + 100000000ull;
        volatile int never = 0;
        for (int f = (g > kHalf ? g - kHalf : 0); f < g; ++f)
          mbar_wait(smem_u32(&bars.full[f % kHalf]), (f / kHalf) & 1, dl2, &never);
        mbar_wait(b_qfull, 0, dl2, &never);
      }
    }
  } else if (warp == 9) {
    // ================================================= MMA issuer ==
    // One thread issues every tcgen05 instruction.  An MMA costs it about
    // as long to issue as the tensor core takes to run it, and the MMA queue
    // is only a few instructions deep, so the loop keeps everything else to
    // the minimum: one wait per K/V pair and per P, one commit per S, per
    // released pair and (at the end) per O, and every shared-memory
    // descriptor precomputed (the loop is unrolled over two turns of the
    // ring's kSlots/2 pairs, so each slot is a constant).  Waits on barriers
    // that have already completed still cost the issuer about 80 cycles each,
    // which is why P is waited for once per tile.
    if (lane == 0) {
      constexpr int kHalf = C::kSlots / 2;
      // a shared-memory descriptor is a fixed high part (layout, strides,
      // swizzle) plus the operand's start address / 16 in its low 14 bits
      const uint64_t hi_s = sdesc_sw128(0, 16, 1024);              // Q and K tiles: K-major
      const uint64_t hi_v = sdesc_sw128(0, C::kPanelBytes, 1024);  // V tiles: MN-major
      const uint32_t q_lo = (sQ & 0x3FFFFu) >> 4, kv_lo = (sKV & 0x3FFFFu) >> 4;
      constexpr uint32_t kTileLo = C::kTileBytes >> 4;
      uint64_t dq[2][C::kQkSteps], dk[kHalf][C::kQkSteps], dv[kHalf][C::kPvSteps];
#pragma unroll
      for (int k = 0; k < C::kQkSteps; ++k) {
        const uint32_t off = ((k >> 2) * C::kPanelBytes + (k & 3) * 32) >> 4;
        dq[0][k] = hi_s | (q_lo + off);
        dq[1][k] = hi_s | (q_lo + kTileLo + off);
#pragma unroll
        for (int u = 0; u < kHalf; ++u) dk[u][k] = hi_s | (kv_lo + ((2 * u + 2) % C::kSlots) * kTileLo + off);
      }
#pragma unroll
      for (int u = 0; u < kHalf; ++u)
#pragma unroll
        for (int k = 0; k < C::kPvSteps; ++k)
          dv[u][k] = hi_v | (kv_lo + ((2 * u + 1) % C::kSlots) * kTileLo + ((k * C::kPvRowsPerStep * 128) >> 4));
      bool ok = mbar_wait(b_qfull, 0, deadline, abort_flag);
      tc_fence_after();
      if (ok && n_it > 0) {
        ok = mbar_wait(smem_u32(&bars.full[0]), 0, deadline, abort_flag);  // group 0: K(0)
        tc_fence_after();
        if (ok) {
          // K(0) sits in slot 0, which is dk[kHalf - 1] ((2 (kHalf - 1) + 2) % kSlots = 0)
          issue_s<D, FP8>(tmem, dq[0], dk[kHalf - 1]);
          mma_commit(smem_u32(&bars.s_full[0]));
          if (two) {
            issue_s<D, FP8>(tmem + 128, dq[1], dk[kHalf - 1]);
            mma_commit(smem_u32(&bars.s_full[1]));
          }
          mma_commit(smem_u32(&bars.empty[0]));
        }
        if constexpr (C::kPsmem) {
          // e4m3: P_i(j) sits in shared-memory buffer j mod 2 of tile i, so the
          // next S only waits until the softmax has read S out of TMEM
          // (s_free): S0(j+1) S1(j+1) PV0(j) PV1(j) per kv tile.  The tensor
          // core computes the next scores while the softmax of this tile runs.
          // S_i(j+1) is issued after PV_i(j-1), so its completion (s_full)
          // also tells the softmax that buffer (j+1) mod 2 is free again.
          uint64_t dp[2][2][C::kPvSteps];
          const uint32_t p_lo = (sP & 0x3FFFFu) >> 4;
          constexpr uint32_t kPLo = C::kPTileBytes >> 4;
#pragma unroll
          for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int bb = 0; bb < 2; ++bb)
#pragma unroll
              for (int k = 0; k < C::kPvSteps; ++k) dp[i][bb][k] = hi_s | (p_lo + (2 * i + bb) * kPLo + 2 * k);
          for (int it0 = 0; ok && it0 < n_it; it0 += 2 * kHalf) {
#pragma unroll
            for (int uu = 0; uu < 2 * kHalf; ++uu) {
              const int u = uu % kHalf, bb = uu & 1;  // it0 is even: buffer = it mod 2
              const int it = it0 + uu;
              if (!ok || it >= n_it) break;
              const bool more = it + 1 < n_it, last = !more;
              const int g = it + 1, bi = g % kHalf;  // group of V(it) and K(it + 1)
              if (!(ok = mbar_wait(smem_u32(&bars.full[bi]), (g / kHalf) & 1, deadline, abort_flag))) break;
              tc_fence_after();
              if (more) {
                if (!(ok = mbar_wait(smem_u32(&bars.s_free[0]), it & 1, deadline, abort_flag))) break;
                tc_fence_after();
                issue_s<D, FP8>(tmem, dq[0], dk[u]);
                mma_commit(smem_u32(&bars.s_full[0]));
                if (two) {
                  if (!(ok = mbar_wait(smem_u32(&bars.s_free[1]), it & 1, deadline, abort_flag))) break;
                  tc_fence_after();
                  issue_s<D, FP8>(tmem + 128, dq[1], dk[u]);
                  mma_commit(smem_u32(&bars.s_full[1]));
                }
              }
              if (!(ok = mbar_wait(smem_u32(&bars.p_full[0][bb]), (it >> 1) & 1, deadline, abort_flag))) break;
              tc_fence_after();
              issue_pv_ss<D, FP8>(tmem + 256, dp[0][bb], dv[u], it > 0);
              if (last) mma_commit(smem_u32(&bars.o_done[0]));
              if (two) {
                if (!(ok = mbar_wait(smem_u32(&bars.p_full[1][bb]), (it >> 1) & 1, deadline, abort_flag))) break;
                tc_fence_after();
                issue_pv_ss<D, FP8>(tmem + 256 + D, dp[1][bb], dv[u], it > 0);
                if (last) mma_commit(smem_u32(&bars.o_done[1]));
              }
              // group g: V(it) and K(it + 1) consumed; its completion also
              // means PV(it) of both tiles is done (the softmax's O rescale)
              if (more) mma_commit(smem_u32(&bars.empty[bi]));
            }
          }
        } else {
        // unrolled over two turns of the ring: the jump back to the loop head
        // costs the issuer about 200 cycles, so it is taken every 2 kHalf steps
        for (int it0 = 0; ok && it0 < n_it; it0 += 2 * kHalf) {
#pragma unroll
          for (int uu = 0; uu < 2 * kHalf; ++uu) {
            const int u = uu % kHalf;
            const int it = it0 + uu;
            if (!ok || it >= n_it) break;
            const bool more = it + 1 < n_it, last = !more;
            const int g = it + 1, bi = g % kHalf;  // group of V(it) and K(it + 1)
            if (!(ok = mbar_wait(smem_u32(&bars.full[bi]), (g / kHalf) & 1, deadline, abort_flag))) break;
            tc_fence_after();
            // O0 += P0 V, then S0 of the next kv tile (it overwrites P0: in order)
            if (!(ok = mbar_wait(smem_u32(&bars.p_full[0][0]), it & 1, deadline, abort_flag))) break;
            tc_fence_after();
            issue_pv<D, FP8>(tmem + 256, tmem, dv[u], it > 0);
            if (last) mma_commit(smem_u32(&bars.o_done[0]));
            if (more) {
              issue_s<D, FP8>(tmem, dq[0], dk[u]);
              mma_commit(smem_u32(&bars.s_full[0]));
            }
            if (two) {
              if (!(ok = mbar_wait(smem_u32(&bars.p_full[1][0]), it & 1, deadline, abort_flag))) break;
              tc_fence_after();
              issue_pv<D, FP8>(tmem + 256 + D, tmem + 128, dv[u], it > 0);
              if (last) mma_commit(smem_u32(&bars.o_done[1]));
              if (more) {
                issue_s<D, FP8>(tmem + 128, dq[1], dk[u]);
                mma_commit(smem_u32(&bars.s_full[1]));
              }
            }
            if (more) mma_commit(smem_u32(&bars.empty[bi]));  // group g: V(it) and K(it + 1) consumed
          }
        }
        }
        if (!ok) record_timeout(p, abort_flag);
      } else if (!ok) {
        record_timeout(p, abort_flag);
      }
      // every issued MMA has completed before TMEM is released
      mma_commit(b_drain);
      volatile int never = 0;
      if (!mbar_wait(b_drain, 0, globaltimer_ns() + p.wait_ns, &never)) record_timeout(p, abort_flag);
    }
  } else {
    // ================================================= softmax + epilogue ==
    const int wg = warp >> 2;            // Q tile 0 or 1
    const int q4 = warp & 3;             // TMEM lane quarter of this warp
    const int row_in_tile = q4 * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t tS = tmem + lane_off + 128 * wg;
    const uint32_t tO = tmem + lane_off + 256 + D * wg;
    // e4m3: this row of the P tile (buffer 0; buffer 1 is kPTileBytes on)
    const uint32_t p_row = sP + 2 * wg * C::kPTileBytes + (row_in_tile >> 3) * 1024 + (row_in_tile & 7) * 128;
    const uint32_t p_r7 = row_in_tile & 7;
    float sl2 = p.scale_log2;
    float vsc = 1.f;
    if (FP8) {
      sl2 *= p.q_scale[h] * p.k_scale[hk];
      vsc = p.v_scale[hk];
    }
    float m_ref = -INFINITY;  // reference max (log2 domain) the current P and O are relative to
    float l_run = 0.f;
    bool ok = true;
    // does this row's own token count as admitted?  (masked-row conventions
    // ULY_ROWS_ZERO and ULY_ROWS_SELF)
    const int lrow = unit_row + wg * kTileRows + row_in_tile;  // row inside the q run
    bool row_valid = true;
    if (p.masked_rows != ULY_ROWS_SDPA && qseg.kv_seg >= 0) {
      const Seg& ks = p.kseg[qseg.kv_seg];
      const int t = lrow / kTileRows;
      if (lrow < ks.len && in_bounds(&g_attn_violations, ks.first + t, 1, p.n_kv_tiles)) {
        const uint4 qb = p.tile_bits[static_cast<int64_t>(b) * p.n_kv_tiles + ks.first + t];
        const int c = lrow % kTileRows;
        const uint32_t w = c < 32 ? qb.x : c < 64 ? qb.y : c < 96 ? qb.z : qb.w;
        row_valid = (w >> (c & 31)) & 1u;
      }
    }
    const bool invert = p.masked_rows == ULY_ROWS_SELF && !row_valid;
    if (wg == 0 || two) {
      // a masked row under ULY_ROWS_SELF reads the complement key sets
      const uint4* active_bits = (invert ? p.active_inv : p.active_bits) + list * p.n_kv_tiles;
      uint4 bits_next = n_it > 0 ? __ldg(active_bits) : make_uint4(0u, 0u, 0u, 0u);
      for (int it = 0; it < n_it; ++it) {
        // the lanes leave together: the TMEM accesses below are warp-collective
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.s_full[wg]), it & 1, deadline, abort_flag))) {
          record_timeout(p, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t a[4][32];
        const uint4 bits = bits_next;
        // a tile whose keys are all admitted for every row of the warp: the
        // TMEM load also takes the row max (tcgen05.ld.red), off the ALU
        const bool full = __all_sync(0xffffffffu, (bits.x & bits.y & bits.z & bits.w) == 0xFFFFFFFFu);
        float mc[4];
        if (full) {
          // (e4m3: two 64-column loads; bf16: four of 32 -- each the form
          // that leaves its kernel's registers unspilled)
          if constexpr (FP8) {
            tmem_ld64_max(tS, a[0], a[1], mc[0]);
            tmem_ld64_max(tS + 64, a[2], a[3], mc[1]);
          } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32_max(tS + 32 * c, a[c], mc[c]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, a[c]);
        }
        if (it + 1 < n_it) bits_next = __ldg(active_bits + it + 1);  // next tile's mask, off the critical path
        tmem_wait_ld();
        if constexpr (C::kPsmem) {
          // S is in registers: the next S may overwrite its TMEM columns
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars.s_free[wg]));
        }
        // (under ULY_ROWS_SELF rows of one warp may see different key sets of
        // the same tile; the masking is per row)
        float m_row;
        if (full) {
          m_row = FP8 ? fmaxf(mc[0], mc[1]) : fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3]));
        } else {
          if ((bits.x & bits.y & bits.z & bits.w) != 0xFFFFFFFFu) mask_tile(a, bits);
          m_row = row_max(a);
        }
        const float m_new = m_row * sl2;
        float alpha = 1.f;
        if (m_new > m_ref + 8.f) {
          alpha = ex2_approx(m_ref - m_new);
          m_ref = m_new;
        }
        // (a row with no admitted key so far keeps m_ref = -inf: use 0 so that
        // masked scores give 2^-inf = 0 rather than NaN)
        // All of S is in registers: P may now overwrite its columns.  P is
        // released to the MMA issuer once all of it and the rescaled running O
        // are stored (the issuer reaches its wait for P later than that, so a
        // release in parts gains nothing).
        const float neg = m_ref == -INFINITY ? 0.f : -m_ref;
        float lsum;
        if constexpr (C::kPsmem)
          lsum = tile_exp_store_e4m3_smem(a, sl2, neg, p_row + (it & 1) * C::kPTileBytes, p_r7);
        else
          lsum = tile_exp_store<0, 2>(a, sl2, neg, tS);
        // (TMEM P: the previous PV has completed, since this S was committed
        // after it; shared-memory P: wait for the K/V group whose release
        // follows PV(it - 1) of both tiles)
        if (it > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          if constexpr (C::kPsmem) {
            constexpr int kHalf = C::kSlots / 2;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.empty[it % kHalf]), (it / kHalf) & 1, deadline,
                                                   abort_flag))) {
              record_timeout(p, abort_flag);
              ok = false;
              break;
            }
            tc_fence_after();
          }
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 16) {
            uint32_t o[16];
            tmem_ld16(tO + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st16(tO + c0, o);
          }
        }
        if constexpr (!C::kPsmem) lsum += tile_exp_store<2, 4>(a, sl2, neg, tS);
        if constexpr (C::kPsmem) fence_proxy_async_smem();  // P's stores -> the MMA (async proxy)
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars.p_full[wg][C::kPsmem ? (it & 1) : 0]));
        l_run = l_run * alpha + lsum;
      }
      // ---- epilogue
      // Ring merge: the running LSE and O rows are loaded before the wait for
      // the last PV, so that their latency hides behind it; the O rows a
      // warp's 32 rows at a time with the lanes along each row (lane l:
      // 16-byte chunk l mod chunks of every 32/chunks-th row), the layout of
      // the output stores below.
      constexpr int kRowBytes = 2 * D, kChunks = kRowBytes / 16;
      constexpr int kRowsPerPass = 32 / kChunks;  // 2 (D = 128) or 4 (D = 64)
      constexpr int kOldVecs = MERGE ? kChunks : 1;
      uint4 old_c[kOldVecs];
      float lse_old = -INFINITY;
      bool old_ok = false;
      if (MERGE && ok) {
        const int sh = p.fused ? 0 : r;
        const int orow_base = qseg.out_row0 < 0 ? p.shard_len[sh] : qseg.out_row0;
        const int oh_ = p.fused ? h : j;
        const bool cols_ok = in_bounds(&g_attn_violations, static_cast<int64_t>(oh_) * D * 2, D * 2, p.out_row_stride);
        const int64_t orow_m = orow_base + lrow;
        if (lrow < qseg.len && cols_ok &&
            in_bounds(&g_attn_violations, orow_m * p.lse_row_stride + oh_, 1, p.lse_batch_stride[sh]) &&
            in_bounds(&g_attn_violations, orow_m * p.out_row_stride, p.out_row_stride, p.out_batch_stride[sh])) {
          old_ok = true;
          lse_old = p.lse[sh][static_cast<int64_t>(b) * p.lse_batch_stride[sh] + orow_m * p.lse_row_stride + oh_];
        }
        const uint8_t* base = p.out[sh] + static_cast<int64_t>(b) * p.out_batch_stride[sh] +
                              static_cast<int64_t>(oh_) * D * 2 + (lane % kChunks) * 16;
#pragma unroll
        for (int i = 0; i < kOldVecs; ++i) {
          const int lr = unit_row + wg * kTileRows + q4 * 32 + i * kRowsPerPass + lane / kChunks;
          const int64_t orow = orow_base + lr;
          old_c[i] = make_uint4(0u, 0u, 0u, 0u);
          if (lr < qseg.len && cols_ok &&
              in_bounds(&g_attn_violations, orow * p.out_row_stride, p.out_row_stride, p.out_batch_stride[sh]))
            old_c[i] = *reinterpret_cast<const uint4*>(base + orow * p.out_row_stride);
        }
      }
      if (ok && n_it > 0) {
        // O is committed once, after the last PV: phase 0
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars.o_done[wg]), 0, deadline, abort_flag))) {
          record_timeout(p, abort_flag);
          ok = false;
        }
        tc_fence_after();
      } else if (ok && !C::kPsmem) {
        // no MMA ran: the Q tile that stages the output below is overwritten
        // only once its load has landed
        if (!__all_sync(0xffffffffu, mbar_wait(b_qfull, 0, deadline, abort_flag))) {
          record_timeout(p, abort_flag);
          ok = false;
        }
      }
      if (ok) {
        const bool store = lrow < qseg.len;
        const bool zero = n_it == 0 || (p.masked_rows == ULY_ROWS_ZERO && !row_valid);
        const float inv = (l_run > 0.f) ? vsc / l_run : 0.f;
        const int orow0 = qseg.out_row0;  // -1: after the image rows of each output shard
        const int ohead = p.fused ? h : j;
        const int shard_lo = (p.fused && qseg.out_shard < 0) ? 0 : (p.fused ? qseg.out_shard : r);
        const int shard_hi = (p.fused && qseg.out_shard < 0) ? p.P : shard_lo + 1;
        // Ring merge (staged path, one output tensor per rank): this call's
        // result joins the running (O, LSE) already in the outputs as in
        // lse_merge_kernel, the new part weighted 1 / (1 + e^(lse_old -
        // lse_new)); a part with LSE -inf leaves the other unchanged, and a
        // row empty in both is written as this call writes it (zero, -inf).
        float w_new = 1.f, lse_w = 0.f;
        bool keep_old = false;
        if (MERGE && store) {
          const float lse_new = row_lse(zero, l_run, m_ref);
          lse_w = lse_new;
          if (old_ok) {
            if (lse_old != -INFINITY) {
              if (lse_new == -INFINITY) {
                keep_old = true;
              } else {
                const float dd = lse_old - lse_new;
                w_new = 1.f / (1.f + ex2_approx(dd * 1.4426950408889634f));
                lse_w = fmaxf(lse_old, lse_new) + log1pf(ex2_approx(-fabsf(dd) * 1.4426950408889634f));
              }
            }
          } else {
            keep_old = true;
          }
        }
        // The output tile goes through shared memory, so that the global
        // stores run along rows (16 lanes a 256-byte row) instead of storing
        // one 16-byte piece of 32 different rows per instruction.  Staging
        // buffer: this tile's Q tile (bf16: every S MMA has completed with
        // the last PV) or its two P buffers (e4m3: every PV has completed);
        // 2D bytes a row, 16-byte chunk c of row r at chunk c ^ (r mod
        // chunks), free of bank conflicts in both directions.  Each warp
        // stages and stores its own 32 rows.
        const uint32_t stage = C::kPsmem ? sP + 2 * wg * C::kPTileBytes : sQ + wg * C::kTileBytes;
        const uint32_t my_row = stage + row_in_tile * kRowBytes;
        const uint32_t sw = row_in_tile & (kChunks - 1);
        const int rt0 = q4 * 32;  // the warp's first row in the tile
        if (MERGE) {
          // the running rows into the staging buffer, where each row's own
          // thread reads them for the merge (and overwrites them with it)
#pragma unroll
          for (int i = 0; i < kOldVecs; ++i) {
            const int rw = i * kRowsPerPass + lane / kChunks;
            const uint4 ov = old_c[i];
            st_shared_v4(stage + (rt0 + rw) * kRowBytes +
                             ((static_cast<uint32_t>(lane % kChunks) ^ static_cast<uint32_t>(rw & (kChunks - 1))) << 4),
                         ov.x, ov.y, ov.z, ov.w);
          }
          __syncwarp();
        }
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          if (n_it > 0) {
            tmem_ld32(tO + c0, o);  // warp-collective: executed whether or not this row is stored
            tmem_wait_ld();
          }
          uint4 v[4];
          uint32_t* vw = reinterpret_cast<uint32_t*>(v);
          if (MERGE && w_new != 1.f && !keep_old) {
            // merge: old + w (new - old) in f32 from the running bf16 row
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint4 ov = ld_shared_v4(my_row + ((static_cast<uint32_t>(c0 / 8 + k) ^ sw) << 4));
              const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int c = 4 * k + e;
                const float x0 = zero ? 0.f : __uint_as_float(o[2 * c]) * inv;
                const float x1 = zero ? 0.f : __uint_as_float(o[2 * c + 1]) * inv;
                const float a0 = __uint_as_float(ow[e] << 16), a1 = __uint_as_float(ow[e] & 0xFFFF0000u);
                vw[c] = pack_bf16x2(fmaf(w_new, x0 - a0, a0), fmaf(w_new, x1 - a1, a1));
              }
            }
          } else {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const float x0 = zero ? 0.f : __uint_as_float(o[2 * c]) * inv;
              const float x1 = zero ? 0.f : __uint_as_float(o[2 * c + 1]) * inv;
              vw[c] = pack_bf16x2(x0, x1);
            }
          }
#pragma unroll
          for (int k = 0; k < 4; ++k)
            st_shared_v4(my_row + ((static_cast<uint32_t>(c0 / 8 + k) ^ sw) << 4), v[k].x, v[k].y, v[k].z, v[k].w);
        }
        __syncwarp();
        // rows of this warp that are not written (a merge that keeps the
        // running row)
        const uint32_t kept = MERGE ? __ballot_sync(0xffffffffu, keep_old) : 0u;
        {
          const int ch = lane % kChunks;
          if (in_bounds(&g_attn_violations, static_cast<int64_t>(ohead) * D * 2, D * 2, p.out_row_stride)) {
            for (int sh = shard_lo; sh < shard_hi; ++sh) {
              const int orow_base = orow0 < 0 ? p.shard_len[sh] : orow0;
              uint8_t* const base = p.out[sh] + static_cast<int64_t>(b) * p.out_batch_stride[sh] +
                                    static_cast<int64_t>(ohead) * D * 2 + ch * 16;
#pragma unroll 4
              for (int i = 0; i < 32; i += kRowsPerPass) {
                const int rw = i + lane / kChunks;  // row of the warp
                const int lr = unit_row + wg * kTileRows + rt0 + rw;  // row inside the q run
                const int64_t orow = orow_base + lr;
                if (lr < qseg.len && !((kept >> rw) & 1u) &&
                    in_bounds(&g_attn_violations, orow * p.out_row_stride, p.out_row_stride, p.out_batch_stride[sh])) {
                  const uint4 val = ld_shared_v4(stage + (rt0 + rw) * kRowBytes +
                                                 ((static_cast<uint32_t>(ch) ^ static_cast<uint32_t>(rw & (kChunks - 1))) << 4));
                  *reinterpret_cast<uint4*>(base + orow * p.out_row_stride) = val;
                }
              }
            }
          }
        }
        if (store && p.lse_out && !keep_old) {
          const float lse = MERGE ? lse_w : row_lse(zero, l_run, m_ref);
          for (int sh = shard_lo; sh < shard_hi; ++sh) {
            const int orow = (orow0 < 0 ? p.shard_len[sh] : orow0) + lrow;
            if (!in_bounds(&g_attn_violations, static_cast<int64_t>(orow) * p.lse_row_stride + ohead, 1,
                           p.lse_batch_stride[sh]))
              continue;
            p.lse[sh][static_cast<int64_t>(b) * p.lse_batch_stride[sh] + static_cast<int64_t>(orow) * p.lse_row_stride +
                      ohead] = lse;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool FP8, bool MERGE>
static cudaError_t launch_one(const AttnParams& p, dim3 grid, cudaStream_t s) {
  using C = Cfg<D, FP8>;
  // the shared-memory limit is a per-device attribute of the function: set
  // it once on every device that launches it (setting it twice is harmless)
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
  if (!bit || !(configured.load(std::memory_order_relaxed) & bit)) {
    e = cudaFuncSetAttribute(attn_kernel<D, FP8, MERGE>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_relaxed);
  }
  attn_kernel<D, FP8, MERGE><<<grid, C::kThreads, C::kSmem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_attention(const AttnParams& p, int D, bool fp8, dim3 grid, cudaStream_t s) {
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
  if (p.merge) {
    if (fp8) return launch_one<128, true, true>(p, grid, s);
    if (D == 128) return launch_one<128, false, true>(p, grid, s);
    return launch_one<64, false, true>(p, grid, s);
  }
  if (fp8) return launch_one<128, true, false>(p, grid, s);
  if (D == 128) return launch_one<128, false, false>(p, grid, s);
  return launch_one<64, false, false>(p, grid, s);
}

// ------------------------------------------------------------ LSE merge --
// Ring-attention merge of two partial results over disjoint key sets
// (flashdreams cp.py ContextParallelAttention._impl_ring):
//   o   = o_a - sigmoid(lse_b - lse_a) * (o_a - o_b)
//   lse = lse_a - logsigmoid(lse_a - lse_b)
// computed in f32 as o_a + w (o_b - o_a), w = 1 / (1 + 2^((lse_a - lse_b)
// log2 e)), lse = max + log(1 + e^-|lse_a - lse_b|); a part with lse = -inf
// leaves the other unchanged.  One thread per 8 bf16 values (16 bytes); the
// threads of a row sit in one warp, so in-place merges are safe.
__global__ void __launch_bounds__(256) lse_merge_kernel(int64_t rows, int D, const uint4* __restrict__ o_a,
                                                        const float* lse_a, const uint4* __restrict__ o_b,
                                                        const float* lse_b, uint4* o_out, float* lse_out) {
  const int per_row = D / 8;
  const int64_t n = rows * per_row;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = i / per_row;
    const float la = lse_a[row], lb = lse_b[row];
    float w, l;
    if (lb == -INFINITY) {
      w = 0.f;
      l = la;
    } else if (la == -INFINITY) {
      w = 1.f;
      l = lb;
    } else {
      const float d = la - lb;
      w = 1.f / (1.f + ex2_approx(d * 1.4426950408889634f));
      l = fmaxf(la, lb) + log1pf(ex2_approx(-fabsf(d) * 1.4426950408889634f));
    }
    const uint4 va = o_a[i], vb = o_b[i];
    const uint32_t* pa = reinterpret_cast<const uint32_t*>(&va);
    const uint32_t* pb = reinterpret_cast<const uint32_t*>(&vb);
    uint4 vo;
    uint32_t* po = reinterpret_cast<uint32_t*>(&vo);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float a0 = __uint_as_float(pa[k] << 16), a1 = __uint_as_float(pa[k] & 0xFFFF0000u);
      const float b0 = __uint_as_float(pb[k] << 16), b1 = __uint_as_float(pb[k] & 0xFFFF0000u);
      po[k] = pack_bf16x2(fmaf(w, b0 - a0, a0), fmaf(w, b1 - a1, a1));
    }
    __syncwarp(__activemask());
    o_out[i] = vo;
    if (i % per_row == 0) lse_out[row] = l;
  }
}

cudaError_t launch_lse_merge(int64_t rows, int D, const void* o_a, const float* lse_a, const void* o_b,
                             const float* lse_b, void* o_out, float* lse_out, int sm_count, cudaStream_t s) {
  const int64_t n = rows * (D / 8);
  if (n <= 0) return cudaSuccess;
  const int64_t want = (n + 255) / 256;
  const int grid = static_cast<int>(want < 8LL * sm_count ? want : 8LL * sm_count);
  lse_merge_kernel<<<grid, 256, 0, s>>>(rows, D, static_cast<const uint4*>(o_a), lse_a,
                                         static_cast<const uint4*>(o_b), lse_b, static_cast<uint4*>(o_out), lse_out);
  return cudaGetLastError();
}

// ------------------------------------------------------------ tile table --
// Per batch: the admitted keys of every 128-key tile of every kv run (bit c
// of tile i of run s = key row0 + 128 i + c, zero past the run's end), and
// the compacted list of tiles with at least one admitted key.  One CTA per
// batch; key order is the global key order (runs in order).
__global__ void __launch_bounds__(1024) tiles_kernel(const __grid_constant__ TileParams p) {
  __shared__ uint4 bits_s[1024];
  __shared__ uint4 inv_s[1024];
  __shared__ int32_t packed_s[1024];
  __shared__ int32_t any_s[1024];
  __shared__ int32_t scan[1024];
  __shared__ int32_t base;
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) base = 0;
  __syncthreads();
  for (int t0 = 0; t0 < p.n_kv_tiles; t0 += 1024) {
    // one warp per tile: lane l decides keys l, l+32, l+64, l+96 (coalesced)
    for (int k = warp; k < 1024; k += 32) {
      const int t = t0 + k;
      if (t >= p.n_kv_tiles) break;
      int s = 0, key0 = 0;
      while (s + 1 < p.n_kseg && t >= p.kseg[s + 1].first) {
        key0 += p.kseg[s].len;
        ++s;
      }
      const int i = t - p.kseg[s].first;
      const int first_key = key0 + i * kTileRows;
      const int n_in = min(kTileRows, p.kseg[s].len - i * kTileRows);
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = lane + 32 * j;
        const int key = first_key + c;
        bool ok = c < n_in && in_bounds(&g_attn_violations, key, 1, p.Nk);
        if (ok && p.key_mask) {
          ok = p.key_mask[static_cast<int64_t>(b) * p.Nk + key] != 0;
        } else if (ok && p.key_ranges) {
          ok = false;
          const int32_t* rg = p.key_ranges + static_cast<int64_t>(b) * p.n_ranges * 2;
          for (int q = 0; q < p.n_ranges; ++q)
            if (key >= rg[2 * q] && key < rg[2 * q + 1]) ok = true;
        }
        w[j] = __ballot_sync(0xffffffffu, ok);
      }
      if (lane == 0) {
        const uint4 wb = make_uint4(w[0], w[1], w[2], w[3]);
        p.tile_bits[static_cast<int64_t>(b) * p.n_kv_tiles + t] = wb;
        bits_s[k] = wb;
        inv_s[k] = make_uint4(~wb.x & lane_mask(n_in, 0), ~wb.y & lane_mask(n_in, 32), ~wb.z & lane_mask(n_in, 64),
                              ~wb.w & lane_mask(n_in, 96));
        packed_s[k] = (s << 20) | i;
        any_s[k] = ((wb.x | wb.y | wb.z | wb.w) != 0u) || (p.all_tiles && n_in > 0);
      }
    }
    __syncthreads();
    // block-wide inclusive scan of "has an admitted key" (Hillis-Steele)
    const int t = t0 + threadIdx.x;
    int any = 0;
    if (t < p.n_kv_tiles) any = any_s[threadIdx.x];
    scan[threadIdx.x] = any;
    __syncthreads();
    for (int off = 1; off < blockDim.x; off <<= 1) {
      const int v = threadIdx.x >= off ? scan[threadIdx.x - off] : 0;
      __syncthreads();
      scan[threadIdx.x] += v;
      __syncthreads();
    }
    if (any && in_bounds(&g_attn_violations, base + scan[threadIdx.x] - 1, 1, p.n_kv_tiles)) {
      const int64_t slot = static_cast<int64_t>(b) * p.n_kv_tiles + base + scan[threadIdx.x] - 1;
      p.active[slot] = packed_s[threadIdx.x];
      p.active_bits[slot] = bits_s[threadIdx.x];
      p.active_inv[slot] = inv_s[threadIdx.x];
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) base += scan[threadIdx.x];
    __syncthreads();
  }
  if (threadIdx.x == 0) p.n_active[b] = base;
  if (p.ring_P > 0) {
    // Ring lists (uly_ring_attention): rank c's list is the batch's list
    // rotated to start at the first tile whose first key lies in c's chunk
    // [ring_bounds[c], ring_bounds[c + 1]) or after it (a tile across a
    // chunk boundary goes with its first key), then the chunks of ranks
    // c + 1, c + 2, ... wrapping around.
    __shared__ int32_t off_s[kMaxRanks];
    const int n = base;
    const int32_t* act = p.active + static_cast<int64_t>(b) * p.n_kv_tiles;
    if (threadIdx.x < p.ring_P) {
      const int bound = p.ring_bounds[threadIdx.x];
      int lo = 0, hi = n;  // first list index whose tile's first key >= bound
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        const int e = act[mid];
        int key0 = 0;
        for (int q = 0; q < (e >> 20); ++q) key0 += p.kseg[q].len;
        if (key0 + (e & 0xFFFFF) * kTileRows < bound)
          lo = mid + 1;
        else
          hi = mid;
      }
      off_s[threadIdx.x] = lo < n ? lo : 0;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < n * p.ring_P; e += blockDim.x) {
      const int c = e / n, k = e - c * n;
      int src = k + off_s[c];
      if (src >= n) src -= n;
      const int64_t from = static_cast<int64_t>(b) * p.n_kv_tiles + src;
      const int64_t to = (static_cast<int64_t>(b) * p.ring_P + c) * p.n_kv_tiles + k;
      p.ring_active[to] = p.active[from];
      p.ring_bits[to] = p.active_bits[from];
      p.ring_inv[to] = p.active_inv[from];
    }
  }
}

cudaError_t launch_tiles(const TileParams& p, cudaStream_t s) {
  tiles_kernel<<<p.B, 1024, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace uly
