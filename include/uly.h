/*
 * uly.h -- C ABI of the GB300 (sm_103a) Ulysses sequence-parallel attention
 * library.  One GPU holds all P "virtual ranks" of a Ulysses group; the
 * library computes, on that GPU, what the P ranks compute together:
 *
 *   uly_to_heads      seq-sharded -> head-sharded exchange (the all-to-all
 *                     is a pure permutation of bytes),
 *   uly_attention     joint text+image attention on the head-sharded layout,
 *   uly_to_seq        head-sharded -> seq-sharded exchange of the output,
 *   uly_sp_attention  the three fused: attention that reads the seq-sharded
 *                     shards directly and writes the seq-sharded output.
 *
 * Sources (web pages, cited by title and section):
 *  [cp]   flashdreams core/attention/cp.py, ContextParallelAttention.
 *         _impl_ulysses: rank r receives heads [r*H/P, (r+1)*H/P) of every
 *         shard, gathered along the sequence in sender-rank order; H must be
 *         divisible by P (ValueError otherwise).
 *  [usp]  sglang multimodal_gen attention/layer.py, USPAttention.forward and
 *         _forward_with_replicated_prefix / _suffix / _kv_prefix: rows every
 *         rank holds (text) stay out of the all-to-all; each rank head-slices
 *         its own copy; a prefix goes before the gathered rows, a suffix after
 *         them; the replicated output is gathered over heads so every shard
 *         receives all heads of those rows; at most one replicated mode per
 *         call (ValueError otherwise).  LocalAttention.forward: the key mask
 *         and GQA (q head h uses kv head h / (Hq/Hkv)).
 *         build_varlen_mask_meta_from_ranges: per-row half-open valid ranges,
 *         ValueError when a range leaves [0, max_seqlen].
 *  [pipe] sglang PR #43521 "pipeline the Ulysses exchange", sections
 *         "Receive slots" (per head group a contiguous
 *         [batch, rows, group_heads, head_dim] slot) and "Automatic group
 *         count" (largest of 7,5,4,3,2 dividing q and k/v heads per rank
 *         while each group still fills four waves of 128-row tiles); the
 *         pipelined result is bit for bit the sequential one.
 *  [lx]   LightX2V PR #1235 "Add optimized Ulysses attention path": the fp8
 *         payload travels with a separate scale tensor.
 *
 * Conventions shared by every entry point:
 *  - Tensors are dense row-major; element sizes: bf16 2 bytes, e4m3 1 byte.
 *    Shard p of q is [B, Rq, Hq, D] and of k/v [B, Rk, Hkv, D] with
 *      NONE:      Rq = Rk = S_l
 *      PREFIX:    Rq = Rk = R + S_l   (rows [0, R) replicated)
 *      SUFFIX:    Rq = Rk = S_l + R   (rows [S_l, S_l + R) replicated)
 *      KV_PREFIX: Rq = S_l, Rk = R + S_l (k/v rows [0, R) replicated)
 *    Rank r's head-sharded tensors are q [B, Nq, Hq/P, D], k/v
 *    [B, Nk, Hkv/P, D] with Nq, Nk the gathered rows: P*S_l image rows in
 *    shard order plus R replicated rows first (PREFIX, and KV_PREFIX for
 *    k/v) or last (SUFFIX).  Row order is the global key order.
 *  - Pointer arguments named q, k, v, o, qh, kh, vh, oh are HOST arrays of
 *    P DEVICE pointers (shard p / rank r), caller-owned, 16-byte aligned.
 *    Every other pointer is a device pointer unless stated.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *    asynchronous: they validate, enqueue kernels and return.  A plan's
 *    device scratch is used by every call made with it, so calls with one
 *    plan must not overlap on the GPU (use one stream per plan).
 *  - The library never allocates memory on the call path; uly_plan_create
 *    allocates the plan's small device scratch once.
 *  - Errors are returned before anything is enqueued, except device-side
 *    wait timeouts, which are recorded on the device and reported by
 *    uly_sync_status.  No call traps, asserts or faults on bad input.
 */
#ifndef ULY_H
#define ULY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define ULY_OK 0
#define ULY_ERR_INVALID 1     /* shapes, divisibility, modes, ranges, NULL or misaligned pointers ([cp], [usp]) */
#define ULY_ERR_UNSUPPORTED 2 /* a valid request this build does not implement (D, dtype combos, P > 16) */
#define ULY_ERR_CUDA 3        /* a CUDA runtime call or kernel launch failed */
#define ULY_ERR_TIMEOUT 4     /* a bounded device wait expired (reported by uly_sync_status) */

/* ---- replicated-row modes ([usp]) --------------------------------------- */
#define ULY_REP_NONE 0
#define ULY_REP_PREFIX 1
#define ULY_REP_SUFFIX 2
#define ULY_REP_KV_PREFIX 3

/* ---- input element types ([lx]); attention output is always bf16 -------- */
#define ULY_BF16 0
#define ULY_E4M3 1

/* ---- what a query row whose own token is a masked key receives ---------- */
#define ULY_ROWS_SDPA 0 /* attention over the admitted keys, as SDPA with a key mask ([usp] LocalAttention) */
#define ULY_ROWS_ZERO 1 /* zero, as the varlen fast path of [usp] USPAttention.forward writes it */
#define ULY_ROWS_SELF 2 /* attention over the masked keys only: the masked rows form a sequence of their own, as the
                           cu_seqlens builders of [lx] make them a separate varlen segment (admitted rows attend to
                           the admitted keys only) */

#define ULY_MAX_RANKS 16

/* Shape of one Ulysses attention call. */
typedef struct uly_desc {
  int32_t B;           /* batch, >= 1 */
  int32_t P;           /* virtual ranks, 1..ULY_MAX_RANKS */
  int32_t S_l;         /* image rows per shard, >= 1 */
  int32_t R;           /* replicated rows (0 iff rep_mode == ULY_REP_NONE) */
  int32_t rep_mode;    /* ULY_REP_* */
  int32_t Hq, Hkv;     /* q and k/v heads; Hq % P == Hkv % P == Hq % Hkv == 0 */
  int32_t D;           /* head dim: 64 or 128 (bf16), 128 (e4m3) */
  int32_t dtype;       /* ULY_BF16 or ULY_E4M3 (q, k, v); outputs are bf16 */
  int32_t masked_rows; /* ULY_ROWS_SDPA, ULY_ROWS_ZERO or ULY_ROWS_SELF */
} uly_desc;

typedef struct uly_plan uly_plan;

/* Validate `desc`, pick the plan's kernels and allocate its device scratch
 * (tile table + status word, a few KB) on `device`.  On success *out is a
 * new plan owned by the caller.  ULY_ERR_INVALID / ULY_ERR_UNSUPPORTED for a
 * bad or unsupported shape, ULY_ERR_CUDA when the allocation fails.  Every
 * call that takes the plan and launches work must be made with `device`
 * current (cudaSetDevice); otherwise it returns ULY_ERR_INVALID before
 * enqueueing anything. */
int uly_plan_create(const uly_desc* desc, int device, uly_plan** out);

/* As uly_plan_create for uneven shards (sglang layer.py passes seq_lens to
 * _usp_input_all_to_all_varlen): shard p holds shard_rows[p] >= 1 image rows
 * (host array of P values) instead of desc->S_l (then ignored).  Gathered
 * image rows are the shards' rows in rank order; shard p's tensors have
 * shard_rows[p] (+ R replicated) rows.  Every entry point except
 * uly_sp_attention_noalloc accepts such a plan. */
int uly_plan_create_varlen(const uly_desc* desc, const int32_t* shard_rows, int device, uly_plan** out);

/* Rows of shard `shard`'s q (is_kv = 0) or k/v (is_kv = 1) tensor, -1 for a
 * bad argument. */
int64_t uly_plan_shard_rows(const uly_plan* plan, int32_t shard, int32_t is_kv);

/* Free a plan (NULL is ignored).  The caller makes sure no call using it is
 * still running on the GPU. */
void uly_plan_destroy(uly_plan* plan);

/* Limit, in nanoseconds, of every device-side wait (default 4e9).  A wait
 * that expires makes the kernel record ULY_ERR_TIMEOUT and return. */
int uly_plan_set_wait_limit(uly_plan* plan, uint64_t ns);

/* Failure-detection test hook: when fill >= 0, the attention kernels' TMA
 * producer never issues K/V copy number `fill` of each CTA (copies count
 * K_0, V_0, K_1, V_1, ...), so the consumer's bounded wait expires and the
 * call reports ULY_ERR_TIMEOUT through uly_sync_status (nothing hangs or
 * faults; the kernels drain and free TMEM).  -1 (the default) disables it.
 * Outputs of a call made with the hook set are undefined. */
int uly_plan_test_withhold_fill(uly_plan* plan, int32_t fill);

/* Checked build (the library compiled with -DULY_CHECKED=1): every index
 * the kernels compute into a global tensor -- a row taken from the segment
 * tables, a head slice, a tile or key index -- is checked against that
 * tensor's extent; an index outside it is counted and its access skipped
 * (no trap, no fault; a skipped K/V copy ends as ULY_ERR_TIMEOUT).
 * uly_checked_violations synchronises the current device and returns the
 * number of violations counted on it since the last reset (and resets the
 * count when reset != 0); -1 in the normal build or on a CUDA error. */
int64_t uly_checked_violations(int32_t reset);

/* Checked-build test hook: the layout kernels' row checks treat the last
 * `rows` rows of every source tensor as outside it (the index arithmetic
 * and the tensors are unchanged, so every access stays inside the real
 * buffers; the runs that the narrowed check rejects are counted and left
 * unwritten).  0 (the default) disables it.  ULY_ERR_UNSUPPORTED in the
 * normal build, ULY_ERR_INVALID for rows < 0. */
int uly_plan_test_check_narrow(uly_plan* plan, int32_t rows);

/* Rows of shard tensors and of the head-sharded tensors (see above).
 * which: 0 = shard q rows, 1 = shard k/v rows (of shard 0 for uneven
 * shards; see uly_plan_shard_rows), 2 = gathered q rows (Nq), 3 = gathered
 * k/v rows (Nk).  Returns -1 for a bad argument. */
int64_t uly_plan_rows(const uly_plan* plan, int which);

/* Automatic head-group count ([pipe] "Automatic group count"): the largest
 * g in {7, 5, 4, 3, 2} dividing both hq_local and hkv_local such that one
 * group still fills four waves of 128-row tiles,
 *     batch_ranks * (hq_local / g) * ceil(q_rows / 128) >= 4 * sm_count,
 * where batch_ranks = B * P (all P ranks share this GPU's SMs) and q_rows is
 * the gathered q rows each rank attends over; 1 when none qualifies.
 * Returns -1 for non-positive arguments. */
int uly_pick_head_groups(int32_t hq_local, int32_t hkv_local, int64_t q_rows, int64_t batch_ranks,
                         int32_t sm_count);

/* Seq-sharded -> head-sharded ([cp] _impl_ulysses; [usp] replicated-row
 * recipes).  Reads shards q[p], k[p], v[p]; writes rank tensors qh[r],
 * kh[r], vh[r]:
 *   qh[r][b, n, j, :] = q[src(n)][b, row(n), r*Hq/P + j, :]
 * and the same for k/v with Hkv; replicated rows are taken from shard r's
 * own copy.  Elements are moved as bytes (bit exact).  Any of the three
 * tensor pairs may be skipped by passing q (or k, or v) as NULL. */
int uly_to_heads(const uly_plan* plan, const void* const* q, const void* const* k, const void* const* v,
                 void* const* qh, void* const* kh, void* const* vh, void* stream);

/* Attention on the head-sharded layout ([usp] LocalAttention.forward /
 * attn_impl.forward over the gathered rows; [pipe] head groups):
 *   for rank r, local q head j (global head h = r*Hq/P + j), batch b, row n:
 *     s_m = scale * <q_n, k_m> over admitted keys m of kv head h / (Hq/Hkv),
 *     oh[r][b, n, j, :] = sum_m softmax(s)_m v_m        (bf16, RNE)
 *   e4m3 inputs: q, k, v are multiplied by q_scale[h], k_scale[h/G],
 *   v_scale[h/G] (device float arrays indexed by GLOBAL head); for bf16 the
 *   scales must be NULL.
 *   Key admission, in global key order (at most one of the two, both NULL
 *   admits every key):
 *     key_mask   device uint8 [B, Nk], nonzero = admitted;
 *     key_ranges device int32 [B, n_ranges, 2] half-open [start, end) ranges
 *                within [0, Nk] ([usp] build_varlen_mask_meta_from_ranges);
 *                ranges outside it are a device-side contract violation that
 *                is clamped, not reported.
 *   A query with no admitted key gets 0.  With ULY_ROWS_ZERO a query row
 *   whose own token is a masked key gets 0.
 *   head_groups: 0 = automatic (uly_pick_head_groups), 1 = every head as
 *   one group, g > 1 = g groups of Hq/(P*g) heads per rank each (g must
 *   divide Hq/P and Hkv/P), processed group after group in one launch (on
 *   one GPU there is no transfer for the groups to overlap with, so the
 *   groups share a launch instead of each paying a partial last wave).
 *   The result is bit-identical for every g.
 *   oh[r] is rank r's [B, Nq, Hq/P, D] bf16 output.
 *   lse: NULL, or a host array of P device pointers to f32 [B, Nq, Hq/P]
 *   (4-byte aligned) that receive each row's log-sum-exp of its admitted
 *   scores, ln sum_m exp(s_m) (the compute_log_sumexp output of the SDPA
 *   calls in flashdreams cp.py); -inf for a row with no admitted key or one
 *   written as zero. */
int uly_attention(uly_plan* plan, const void* const* qh, const void* const* kh, const void* const* vh,
                  const uint8_t* key_mask, const int32_t* key_ranges, int32_t n_ranges, float scale,
                  int32_t head_groups, const float* q_scale, const float* k_scale, const float* v_scale,
                  void* const* oh, float* const* lse, void* stream);

/* Head-sharded -> seq-sharded for the bf16 output ([cp] output exchange;
 * [usp] replicated output gathered over heads):
 *   o[p][b, row, h, :] = oh[h / (Hq/P)][b, n(p, row), h % (Hq/P), :]
 * where replicated rows map to the same gathered row for every p.  Bit exact. */
int uly_to_seq(const uly_plan* plan, const void* const* oh, void* const* o, void* stream);

/* Fused exchange + attention + exchange: the same result as uly_to_heads,
 * uly_attention and uly_to_seq in sequence (bit-identical to it), read
 * straight from the shards q[p], k[p], v[p] and written straight to the
 * bf16 shard outputs o[p] [B, Rq, Hq, D], with no staging copy.  Arguments
 * as in uly_attention; lse, when given, is per shard f32 [B, Rq, Hq]
 * (replicated rows' values reach every shard, like their outputs).
 * The call enqueues work only (no host synchronisation), so it may be
 * captured into a CUDA graph; the graph keeps the pointers, so replays read
 * the buffers' current values.  Make the first call for a plan outside a
 * capture (it sets the kernel's shared-memory limit on the device).
 * uly_sp_attention_host may be captured the same way. */
int uly_sp_attention(uly_plan* plan, const void* const* q, const void* const* k, const void* const* v,
                     const uint8_t* key_mask, const int32_t* key_ranges, int32_t n_ranges, float scale,
                     int32_t head_groups, const float* q_scale, const float* k_scale, const float* v_scale,
                     void* const* o, float* const* lse, void* stream);

/* Staged path with the exchange pipelined against the attention (sglang
 * PR #43521, "Motivation": while one group attends, the next group's q/k/v
 * moves; finished groups send their output back while later groups still
 * attend).  The pipeline's chunks are the ranks' heads, the first rank
 * starting with chunks of 1, 2 and 4 head groups and the last head group of
 * the last rank a chunk of its own, so that little exchange is exposed
 * before the first launch and after the last.  Each
 * chunk's seq -> heads exchange is the gather kernel of uly_to_heads
 * restricted to that rank and head range, queued on `copy_stream` (its CTAs
 * fit on the SMs beside the attention CTAs); each chunk attends as soon as
 * its inputs are in place, and its output goes back by the uly_to_seq
 * gather on `copy_stream` while later chunks attend.  The result is
 * bit-identical to uly_to_heads + uly_attention + uly_to_seq (and to
 * uly_sp_attention).
 *   q, k, v, o: shard tensors as in uly_sp_attention;
 *   qh, kh, vh, oh: caller-owned staging (rank tensors as in uly_to_heads /
 *   uly_attention); head_groups as in uly_attention.
 *   copy_stream must be a non-NULL stream other than `stream` (created
 *   non-blocking, or the legacy default stream serialises the two).  The
 *   chunks' attention alternates between two streams owned by the plan
 *   (created on first use), so that one chunk's last wave overlaps the next
 *   chunk's first.  The call orders all of them with events so that work
 *   already queued on `stream` comes first and `stream` is ordered after the
 *   last exchange back. */
int uly_pipelined_attention(uly_plan* plan, const void* const* q, const void* const* k, const void* const* v,
                            void* const* qh, void* const* kh, void* const* vh, void* const* oh,
                            const uint8_t* key_mask, const int32_t* key_ranges, int32_t n_ranges, float scale,
                            int32_t head_groups, const float* q_scale, const float* k_scale, const float* v_scale,
                            void* const* o, void* stream, void* copy_stream);

/* uly_sp_attention with the shards in host memory: copies the inputs in,
 * attends, and copies the output out, overlapping the three.  Every rank's
 * heads form one chunk, except that the first rank starts with chunks of
 * 1, 2 and 4 head groups and the last head group of the last rank is a
 * chunk of its own, so that little copying is exposed before the first
 * launch and after the last: the copy engines move
 * chunk c+1's input heads (every shard's rows, one pitched copy per shard
 * and tensor) while the SMs attend chunk c, and chunk c's output heads go
 * back while later chunks attend.  (Host memory sits across the PCIe /
 * chip-to-chip link from the GPU just as, in the pages' multi-GPU setting,
 * the other ranks' shards sit across the interconnect; splitting by rank
 * keeps most copied runs H/P * D elements long.)  The first chunk's copy in
 * (exposed: nothing runs before it) and the last chunk's copy out are done
 * by a copy kernel instead when every host buffer involved is page-locked
 * memory mapped into the device's address space (as cudaHostAlloc memory is
 * on a 64-bit system) and 16-byte aligned: its rows are narrow, which the
 * copy engine moves at about half the link's rate.  The output is
 * bit-identical to uly_sp_attention on the same device tensors.
 *   q_host, k_host, v_host: P host pointers to shard tensors laid out as in
 *     uly_sp_attention; page-locked (cudaHostAlloc / cudaHostRegister) for
 *     the copies to overlap -- pageable memory gives the same result without
 *     the overlap.
 *   q, k, v: P device shard tensors the call fills (caller-owned staging;
 *     16-byte aligned), o: P device output shard tensors (filled as well),
 *   o_host: P host pointers receiving the output shards.
 *   Other arguments as in uly_sp_attention (key_mask / key_ranges and the
 *   fp8 scales are device memory; no LSE output).
 * Work runs on four streams owned by the plan (created on first use): the
 * call orders them after the work already queued on `stream`, and `stream`
 * after the last copy out, so the host buffers may be read once `stream` has
 * been synchronised.  The plan's tile table is in use until then: calls
 * with the same plan must be ordered on one stream.  ULY_ERR_INVALID for
 * NULL host pointers and as uly_sp_attention. */
int uly_sp_attention_host(uly_plan* plan, const void* const* q_host, const void* const* k_host,
                          const void* const* v_host, void* const* q, void* const* k, void* const* v,
                          const uint8_t* key_mask, const int32_t* key_ranges, int32_t n_ranges, float scale,
                          int32_t head_groups, const float* q_scale, const float* k_scale, const float* v_scale,
                          void* const* o, void* const* o_host, void* stream);

/* Ring-attention merge of two attention results of the same query rows over
 * disjoint key sets (flashdreams cp.py ContextParallelAttention._impl_ring):
 *   o   = o_a - sigmoid(lse_b - lse_a) * (o_a - o_b)
 *   lse = lse_a - logsigmoid(lse_a - lse_b)
 * o_a, o_b, o_out: device bf16 [rows, D] (D = 64 or 128, 16-byte aligned);
 * lse_a, lse_b, lse_out: device f32 [rows].  A part whose lse is -inf (no
 * admitted key) leaves the other unchanged.  o_out / lse_out may be o_a /
 * lse_a (in place).  Merging the results of attention over consecutive key
 * ranges (uly_attention with key_ranges, one range per virtual ring rank)
 * gives attention over all of them.  ULY_ERR_INVALID for bad sizes, NULL or
 * misaligned pointers. */
int uly_lse_merge(int64_t rows, int32_t D, const void* o_a, const float* lse_a, const void* o_b,
                  const float* lse_b, void* o_out, float* lse_out, void* stream);

/* One ring step with the merge fused into the attention's epilogue: the
 * attention of uly_attention over the admitted keys (one virtual ring rank's
 * key chunk) is merged into the running result (oh, lse) that earlier steps
 * left, with the weights of uly_lse_merge, instead of being written to its
 * own buffers and merged by a separate pass (which reads and writes the
 * output twice more).  On entry oh[r] / lse[r] hold the running result of
 * the earlier chunks; a row whose lse is -inf counts as empty (its oh
 * values are not read).  Start a ring by filling lse with -inf or by a first
 * uly_attention call with the lse output.  A row with no admitted key in
 * this chunk keeps its running values; a row empty in both is written as
 * uly_attention writes it (zero, -inf).  The merged O is rounded to bf16
 * once per step from f32, so a chain of steps equals the separate merges up
 * to rounding.  Arguments as in uly_attention, with lse required (f32
 * [B, Nq, Hq/P] per rank, read and written).  ULY_ERR_INVALID for a NULL
 * lse and as uly_attention. */
int uly_attention_merge(uly_plan* plan, const void* const* qh, const void* const* kh, const void* const* vh,
                        const uint8_t* key_mask, const int32_t* key_ranges, int32_t n_ranges, float scale,
                        int32_t head_groups, const float* q_scale, const float* k_scale, const float* v_scale,
                        void* const* oh, float* const* lse, void* stream);

/* Ring attention over the P virtual ring ranks in one launch (flashdreams
 * cp.py ContextParallelAttention._impl_ring): virtual rank c holds the key
 * chunk [chunk_bounds[c], chunk_bounds[c + 1]) of the global key order, and
 * the queries of rank r take the chunks in the order that function visits
 * them -- r's own first, then r + 1, r + 2, ... (mod P).  The merge of each
 * chunk's partial result into the running one (the sigmoid / logsigmoid
 * update of uly_lse_merge) is carried out on chip as the online softmax's
 * rescale, in f32 (the function's convert_to_fp32 option), so O is rounded
 * to bf16 once, at the end.  The result is attention over all admitted keys
 * and equals the chain uly_attention + uly_attention_merge (or +
 * uly_lse_merge) over the chunks up to rounding.  Keys go in 128-key tiles:
 * a tile that straddles a chunk boundary is taken with the chunk of its
 * first key.
 * chunk_bounds: host array of P + 1 int32, chunk_bounds[0] = 0,
 * non-decreasing, chunk_bounds[P] = the plan's gathered key rows
 * (uly_plan_rows(plan, 3), Nk).  Other arguments and the outputs (oh, and lse
 * if not NULL) as in uly_attention.  ULY_ERR_INVALID for NULL or bad
 * chunk_bounds and as uly_attention. */
int uly_ring_attention(uly_plan* plan, const void* const* qh, const void* const* kh, const void* const* vh,
                       const uint8_t* key_mask, const int32_t* key_ranges, int32_t n_ranges,
                       const int32_t* chunk_bounds, float scale, int32_t head_groups, const float* q_scale,
                       const float* k_scale, const float* v_scale, void* const* oh, float* const* lse,
                       void* stream);

/* Allocation-free fused attention.  The source pages have no counterpart:
 * this entry point exists for callers that cannot call cudaMalloc -- an
 * application whose device memory belongs to its own pool (a framework's
 * caching allocator, a serving runtime that reserves the GPU's memory up
 * front) cannot let a library allocate behind it: the allocation escapes
 * the pool's accounting, can fail when the pool already holds the memory,
 * and cudaMalloc/cudaFree synchronize the device.  uly_plan_create
 * allocates, so such callers use this call, which needs no plan.
 *
 * It computes exactly what uly_sp_attention computes for a plan made from
 * `desc` (same kernels, same bytes), with arguments as there.  Its scratch
 * (the kv tile table and a status word) is a fixed device array inside the
 * library, 224 KB + 256 bytes, that every GPU which loads the library holds
 * until the process exits:
 *  - the call rejects, with ULY_ERR_UNSUPPORTED and before enqueueing
 *    anything, a shape whose B * ceil-tiles of 128 keys over all kv runs
 *    exceeds 4096 (about 512K keys at B = 1);
 *  - every call looks up the array's device address in the current
 *    device's context (cudaGetSymbolAddress, a host-side lookup that
 *    allocates nothing), so the call stays valid after the context has been
 *    torn down and created again;
 *  - with lazy module loading (the CUDA default), the first call on a
 *    device loads the library's kernels and creates the array on that
 *    device: memory that the driver allocates outside the caller's pool.
 *    Make that first call during warm-up, before the pool reserves the
 *    device's memory and before any stream capture;
 *  - every call shares the one array and leaves its contents behind: the
 *    call clears what must start at zero itself, but calls that overlap on
 *    the GPU (two streams, or two threads) race on it and must not be used;
 *  - device wait timeouts are recorded in the array's status word, which
 *    uly_noalloc_sync_status reads back and clears (each call of this
 *    entry point clears it first, so read it before the next call).
 * It allocates no device memory and calls no allocating CUDA or library
 * routine. */
int uly_sp_attention_noalloc(const uly_desc* desc, const void* const* q, const void* const* k,
                             const void* const* v, const uint8_t* key_mask, const int32_t* key_ranges,
                             int32_t n_ranges, float scale, int32_t head_groups, const float* q_scale,
                             const float* k_scale, const float* v_scale, void* const* o, float* const* lse,
                             void* stream);

/* The status of uly_sp_attention_noalloc calls (no counterpart on the source
 * pages, like that call): synchronize `stream`, then read and clear the
 * status word in the allocation-free call's device array.  Returns ULY_OK,
 * ULY_ERR_TIMEOUT when a device wait of such a call expired since the
 * word was last cleared, or ULY_ERR_CUDA.  Allocates nothing. */
int uly_noalloc_sync_status(void* stream);

/* Synchronize `stream`, then read and clear the plan's device status word.
 * Returns ULY_OK, ULY_ERR_TIMEOUT when a device wait expired since the last
 * check, or ULY_ERR_CUDA when the stream reports an error. */
int uly_sync_status(uly_plan* plan, void* stream);

/* Static text for a status code. */
const char* uly_status_string(int status);

/* Number of SMs of `device` (for uly_pick_head_groups), or -1. */
int32_t uly_device_sm_count(int device);

#ifdef __cplusplus
}
#endif

#endif /* ULY_H */
