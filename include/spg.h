/*
 * spg.h — C ABI of the query-aware sparse-page decode attention library
 * (libspg.so, hand-written CUDA for sm_103a).
 *
 * One decode step over a paged KV cache:
 *   1. keep per-page metadata current when a token is appended
 *      (Quest 完全拆解, 关键性估计算法: M_i <- max(M_i, k_i), m_i <- min(m_i, k_i);
 *       SALS长序列推理优化, 算法简介: the low-rank index-key preprocessing),
 *   2. score every candidate page against the current query
 *      (Quest 核心机制: sum_i max(q_i m_i, q_i M_i);  SALS Quant Sals Indexer:
 *       int4 low-rank index key, dequantise, block log-sum-exp),
 *   3. take the exact top-k pages, lower page index winning ties, plus forced
 *      sink / recent (tail) pages (SALS QSI Top-k 计算实现; Day 10·2 sparse top-k
 *      块选择, 确定性红线), writing only int32 page ids (SequenceO1 close
 *      reading §3.3, the select -> attend two-kernel boundary),
 *   4. run split-K flash-decoding over the selected pages only and merge the
 *      splits by log-sum-exp (SALS SFAA 四阶段 flow; AICPU Tiling challenge 2).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers, 16-byte aligned, contiguous
 *     row-major in the layouts stated below; the caller owns all memory.
 *     The library never allocates device memory.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and never synchronise, except spg_read_device_error.
 *   - Nothing throws across the ABI.  Host-side checks return SPG_EINVAL
 *     (bad sizes, null or misaligned pointers), SPG_EUNSUPPORTED (valid but
 *     not built: e.g. head_dim outside {64, 128}), SPG_EWORKSPACE (workspace
 *     too small) before anything is launched; a failed launch is SPG_ECUDA.
 *   - Faults the device can see (a page-table entry outside the pool, a
 *     seq_len beyond the page table, a selected page id out of range, a
 *     bounded wait that ran out) are not dereferenced: the offending page is
 *     skipped and a bit (SPG_DEVERR_*) is OR-ed into the error word at the
 *     start of the workspace.  spg_read_device_error() fetches it.
 *   - The workspace must be zero-filled once after allocation; the library
 *     leaves its bookkeeping in a reusable state after every call.  After a
 *     call that reported SPG_DEVERR_TIMEOUT, zero it again before reuse.
 *     Calls that share a workspace must not overlap on the GPU (order them
 *     on one stream).
 *
 * Shapes (B batch, Hq / Hkv query / kv heads, G = Hq / Hkv, d head_dim,
 * S page_size, P_phys num_phys_pages, MP max_pages_per_seq,
 * n_sel = token_budget / page_size, ds sketch_dim):
 *   q            [B][Hq][d]            q_dtype (fp16 | bf16); query head j
 *                                      belongs to kv-head j / G
 *   k_pool,v_pool[P_phys][Hkv][S][d]   kv_dtype (fp16 | bf16 | int8)
 *   k_scale,v_scale [P_phys][Hkv][S]   fp16, per-token per-head dequant
 *                                      scales (int8 pools only, else NULL)
 *   page_table   [B][MP] int32         physical page of each logical page
 *   seq_lens     [B] int32             tokens in each sequence, counting the
 *                                      token appended this step
 *   minmax       [B][Hkv][MP][2][d]    kv_dtype (q_dtype for int8 pools);
 *                                      per sequence, kv-head and LOGICAL
 *                                      page: [..][0][:] = per-channel min m,
 *                                      [..][1][:] = max M of K over the
 *                                      page's valid tokens (Quest); for int8
 *                                      pools the min / max of the dequantised
 *                                      keys code * scale, rounded outward (m
 *                                      down, M up) to the 16-bit type
 *   sketch       [B][Hkv][MP][S][ds/2] uint8, per logical block; int4 codes
 *                                      of the projected keys, two's
 *                                      complement, channel 2j in the low
 *                                      nibble of byte j (sketch)
 *   sketch_scale [B][Hkv][MP] fp32     one dequant scale per block (sketch)
 * Page metadata is kept in logical page order per sequence (not per physical
 * page) so that scoring one (sequence, kv-head) reads a single contiguous
 * range and needs no page-table lookup.
 *   proj         [d][ds] fp32          fixed projection P shared by all heads
 *   scores       [B][Hkv][MP] fp32     page scores; -inf for pages that are
 *                                      not candidates
 *   sel          [B][Hkv][n_sel] int32 selected logical page ids, ascending;
 *                                      unused tail entries are -1
 *   sel_cnt      [B][Hkv] int32        number of valid entries in sel
 *   out          [B][Hq][d] fp32       attention output
 *   lse          [B][Hq] fp32          natural-log log-sum-exp of the scaled
 *                                      logits over the attended tokens
 *                                      (may be NULL)
 * A sequence with seq_len 0 gets out = 0 and lse = -inf.
 */
#ifndef SPG_H_
#define SPG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* spg_stream_t; /* a cudaStream_t */

#define SPG_ABI_VERSION 2

typedef enum {
  SPG_OK = 0,
  SPG_EINVAL = 1,
  SPG_EUNSUPPORTED = 2,
  SPG_ECUDA = 3,
  SPG_EWORKSPACE = 4
} spg_status;

typedef enum {
  SPG_SEL_QUEST = 0,       /* per-page per-channel min/max upper bound */
  SPG_SEL_SKETCH_INT4 = 1, /* int4 low-rank index key, block log-sum-exp */
  SPG_SEL_ALL = 2,         /* every page (dense attention) */
  SPG_SEL_PROBE = 3        /* largest q.k over a few sampled keys of each page */
} spg_selector;

typedef enum { SPG_F16 = 0, SPG_BF16 = 1, SPG_I8 = 2 } spg_dtype;

/* device error bits, OR-ed into the workspace error word */
#define SPG_DEVERR_PAGE_ID 1 /* page-table entry outside [0, num_phys_pages) */
#define SPG_DEVERR_SEQ_LEN 2 /* seq_lens[b] < 0 or > max_pages_per_seq * page_size */
#define SPG_DEVERR_SEL 4     /* sel entry outside [0, P_b) or sel_cnt outside [0, n_sel] */
#define SPG_DEVERR_TIMEOUT 8 /* a bounded wait for an asynchronous copy ran out */

typedef struct spg_params {
  int32_t batch;             /* B >= 1 */
  int32_t num_q_heads;       /* Hq, a multiple of num_kv_heads, G = Hq/Hkv in {1,2,4,8} */
  int32_t num_kv_heads;      /* Hkv >= 1 */
  int32_t head_dim;          /* d in {64, 128} */
  int32_t page_size;         /* S: 16, 32, 64 or 128 tokens (a SALS block); 8 is
                                valid but not built (SPG_EUNSUPPORTED), and so is a
                                page whose K + V (+ int8 scales) of one kv-head
                                exceed 34 KB (fp16/bf16 at d = 128: S <= 64) */
  int32_t num_phys_pages;    /* P_phys: pages in the pool */
  int32_t max_pages_per_seq; /* MP: columns of page_table */
  int32_t kv_dtype;          /* spg_dtype */
  int32_t q_dtype;           /* SPG_F16 or SPG_BF16; equal to kv_dtype unless kv is int8 */
  int32_t selector;          /* spg_selector */
  int32_t token_budget;      /* tokens attended per (batch, kv-head), forced pages
                                included; a multiple of page_size; ignored by SPG_SEL_ALL */
  int32_t n_sink_pages;      /* pages [0, n_sink) always attended */
  int32_t n_recent_pages;    /* last n_recent pages always attended; the sketch
                                selector needs >= 1 (the open tail block) */
  int32_t sketch_dim;        /* ds = 16 for SPG_SEL_SKETCH_INT4, else ignored */
  float softmax_scale;       /* 0 => 1/sqrt(head_dim) */
  /* Adaptive budget (SequenceO1 close reading §3.2 / §4.2: keep the leading
   * pages whose cumulative softmax mass of page scores reaches top_p).  0 =
   * off: the token budget fixes the count.  In (0, 1]: of the candidates,
   * in (score desc, page asc) order, keep the smallest prefix whose share
   * of exp(tau * (s - max s)) over all candidates reaches top_p (tau = 1
   * for the sketch selector, whose score is a log block mass; the softmax
   * scale for Quest), at least min(min_pages, cap) and at most the cap
   * n_sel - forced pages.  Weights and sums in fp32, in a fixed order.
   * Needs n_sel <= 1024 (SPG_EUNSUPPORTED beyond); ignored by SPG_SEL_ALL. */
  float top_p;
  int32_t min_pages;         /* adaptive budget: fewest candidate pages kept (>= 0) */
  /* Probe selector (Day 10·2 sparse top-k, §1-§2): a page's score is the
   * largest q . k (max also over the group's query heads) over n_probe of
   * its tokens, sampled from its first token in steps of max(valid tokens /
   * n_probe, 1).  0 => 8.  The probe selector has no metadata: it reads the
   * keys, so the `minmax` argument of every entry point is the K pool for it
   * (and sparse_page_meta_update has nothing to do).  fp16/bf16 pools only. */
  int32_t n_probe;
} spg_params;

/* Library ABI version (SPG_ABI_VERSION of the build). */
int32_t spg_abi_version(void);

/* Static text for a status code. */
const char* spg_status_str(int32_t status);

/* Host-only check of a parameter block: SPG_OK, SPG_EINVAL or SPG_EUNSUPPORTED. */
spg_status spg_validate(const spg_params* p);

/* Bytes of device workspace every entry point needs for these parameters
 * (the same figure for all of them).  Host only. */
spg_status spg_workspace_size(const spg_params* p, size_t* bytes);

/* Metadata maintenance (Quest 关键性估计算法, insert-time update; SALS low-rank
 * preprocessing).
 * rebuild == 0 (append): for each sequence the token at position
 *   seq_lens[b]-1 has just been written to the pools.  Quest: its page's
 *   min/max is updated (the page's first token starts them afresh).
 *   Sketch: when that token completes a block, the block's S keys are
 *   dequantised, projected through proj and quantised to int4 with one scale.
 * rebuild != 0: the metadata of every page of every sequence is rebuilt from
 *   the pool (Quest: every page; sketch: every full block).
 * Quest needs minmax (sketch args may be NULL); the sketch selector needs
 * sketch, sketch_scale and proj (minmax may be NULL); k_scale for int8. */
spg_status sparse_page_meta_update(const spg_params* p, const void* k_pool, const void* k_scale,
                                   const int32_t* page_table, const int32_t* seq_lens,
                                   int32_t rebuild, void* minmax, uint8_t* sketch,
                                   float* sketch_scale, const float* proj, void* ws,
                                   size_t ws_bytes, spg_stream_t stream);

/* Page scores of every candidate page (Quest 核心机制; SALS QSI steps 1-3).
 * Candidates of sequence b are pages [n_sink, P_b - n_recent); every other
 * entry of the [B][Hkv][MP] array is -inf.  Quest: the largest over the
 * group's query heads of sum_i max(q_i m_i, q_i M_i).  Sketch: with the
 * group-mean query projected and quantised to int8 codes qc (scale sq),
 * z_t = (sum_j qc_j kc_tj) * sq * sk_block / sqrt(d) and the block score is
 * log sum_t exp(z_t). */
spg_status sparse_page_score(const spg_params* p, const void* q, const int32_t* page_table,
                             const int32_t* seq_lens, const void* minmax, const uint8_t* sketch,
                             const float* sketch_scale, const float* proj, float* scores, void* ws,
                             size_t ws_bytes, spg_stream_t stream);

/* Score + exact top-k (SALS QSI steps 1-5; Quest Top-K filtering).  Per
 * (batch, kv-head): forced pages F = [0, n_sink) U [P_b - n_recent, P_b);
 * the k_top = n_sel - |F| best candidates by (score desc, page asc); sel =
 * F U top-k in ascending order, sel_cnt = its size (all pages when
 * P_b <= n_sel). */
spg_status sparse_page_select(const spg_params* p, const void* q, const int32_t* page_table,
                              const int32_t* seq_lens, const void* minmax, const uint8_t* sketch,
                              const float* sketch_scale, const float* proj, int32_t* sel,
                              int32_t* sel_cnt, void* ws, size_t ws_bytes, spg_stream_t stream);

/* The sketch selector's integer arithmetic, for checking it exactly (SALS
 * 长序列推理优化, Quant Sals Indexer steps 1-2: the int4 index key times the
 * int8 index query as an integer matrix product, before any dequantisation).
 * Per (batch, kv-head) unit, with the same device routines the decode step's
 * scan uses:
 *   qc   [B][Hkv][16] int32  the int8 index-query codes (group-mean query
 *                            projected through proj, scale max|q~|/127,
 *                            round half to even), one code per int32
 *   sq   [B][Hkv] fp32       the index-query scale
 *   dots [B][Hkv][MP][S] int32  for every token t of every candidate block
 *                            p in [n_sink, P_b - n_recent): sum_j qc_j *
 *                            code_{p,t,j}, exact; every other entry is 0
 * Sketch selector only (SPG_EINVAL otherwise); sketch holds the int4 codes
 * of sparse_page_meta_update.  Device-detected faults go to the workspace
 * error word. */
spg_status sparse_page_sketch_dots(const spg_params* p, const void* q, const int32_t* seq_lens,
                                   const uint8_t* sketch, const float* proj, int32_t* qc,
                                   float* sq, int32_t* dots, void* ws, size_t ws_bytes,
                                   spg_stream_t stream);

/* Flash-decoding over the selected pages only (SALS SFAA; Quest
 * Approximate attention): for query head j of kv-head h, attention over
 * the tokens t < seq_lens[b] of pages sel[b][h][0..sel_cnt), softmax
 * renormalised over them (Day 10·2: the softmax covers the selected blocks
 * only).  int8 K/V are dequantised by their per-token scales. */
spg_status sparse_decode_attention(const spg_params* p, const void* q, const void* k_pool,
                                   const void* v_pool, const void* k_scale, const void* v_scale,
                                   const int32_t* page_table, const int32_t* seq_lens,
                                   const int32_t* sel, const int32_t* sel_cnt, float* out,
                                   float* lse, void* ws, size_t ws_bytes, spg_stream_t stream);

/* sparse_page_select followed by sparse_decode_attention, one call; for the
 * Quest and sketch selectors with page tables of at most 8192 pages both run
 * in a single launch (see sparse_decode_step); the probe selector takes its
 * selection launch and the attention launch. */
spg_status sparse_decode_select_attend(const spg_params* p, const void* q, const void* k_pool,
                                       const void* v_pool, const void* k_scale,
                                       const void* v_scale, const int32_t* page_table,
                                       const int32_t* seq_lens, const void* minmax,
                                       const uint8_t* sketch, const float* sketch_scale,
                                       const float* proj, int32_t* sel, int32_t* sel_cnt,
                                       float* out, float* lse, void* ws, size_t ws_bytes,
                                       spg_stream_t stream);

/* The whole decode step in one call: the metadata update for the token just
 * appended at seq_lens[b]-1 (as sparse_page_meta_update with rebuild == 0),
 * then sparse_decode_select_attend.  Where the parameters allow it (Quest or
 * sketch selector, page tables of at most 8192 pages), selection and
 * attention run as one launch of one thread-block cluster of up to 8 CTAs per
 * (batch, kv-head) (4 or 2 when the units would not fit one wave), or as one
 * persistent launch with task queues (spg_step_kernel says which); with
 * n_recent_pages >= 1 (and sketch_dim 16 for the sketch selector) the append
 * runs inside that launch too (the appended token's page is forced, so no
 * scoring depends on it). */
spg_status sparse_decode_step(const spg_params* p, const void* q, const void* k_pool,
                              const void* v_pool, const void* k_scale, const void* v_scale,
                              const int32_t* page_table, const int32_t* seq_lens, void* minmax,
                              uint8_t* sketch, float* sketch_scale, const float* proj,
                              int32_t* sel, int32_t* sel_cnt, float* out, float* lse, void* ws,
                              size_t ws_bytes, spg_stream_t stream);

/* Dense flash-decoding over every page of every sequence (the baseline the
 * Quest page compares against: the full KV read). */
spg_status dense_decode_attention(const spg_params* p, const void* q, const void* k_pool,
                                  const void* v_pool, const void* k_scale, const void* v_scale,
                                  const int32_t* page_table, const int32_t* seq_lens, float* out,
                                  float* lse, void* ws, size_t ws_bytes, spg_stream_t stream);

/* Bytes of the library-owned scratch array behind
 * sparse_decode_attention_noalloc (16 MiB).  A call needs
 * 256 + 4 * units + 512 * rows * (head_dim + 2) bytes (each region rounded
 * up to 256), rows = batch * num_q_heads, units = batch * num_kv_heads: at
 * most 252 rows at head_dim 128, 496 at 64. */
#define SPG_NOALLOC_SCRATCH_BYTES (16u << 20)

/* sparse_decode_attention for callers that cannot allocate device memory
 * (no counterpart in the source papers: it exists for embedding this
 * library).  Plugins run by a host framework that owns all device memory
 * and gives them no allocator or workspace, and serving loops that forbid
 * cudaMalloc after start-up, cannot supply the workspace the other entry
 * points take.  This one takes the same arguments minus the workspace and
 * keeps its scratch (split partials, an error word) in one array of
 * SPG_NOALLOC_SCRATCH_BYTES of device memory owned by the library, which
 * every GPU that loads the library holds until the process exits.
 * - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 * - The first call on a device, with that device current, looks up the
 *   array's device address (cudaGetSymbolAddress) and caches it; make that
 *   first call before any stream capture.
 * - Returns SPG_EWORKSPACE when the problem's partials do not fit the array
 *   (see SPG_NOALLOC_SCRATCH_BYTES), before launching anything.
 * - All calls on a device share the array and leave their contents in it:
 *   calls whose kernels overlap on the GPU (unordered streams) race and
 *   corrupt each other's results.  Order them on one stream.
 * - Device-detected faults (bad page ids) are skipped as in the other entry
 *   points, but this entry point has no error word the caller can read. */
spg_status sparse_decode_attention_noalloc(const spg_params* p, const void* q, const void* k_pool,
                                           const void* v_pool, const void* k_scale,
                                           const void* v_scale, const int32_t* page_table,
                                           const int32_t* seq_lens, const int32_t* sel,
                                           const int32_t* sel_cnt, float* out, float* lse,
                                           spg_stream_t stream);

/* Short-sequence dense bypass (Quest 完全拆解, 短序列的负收益: the read ratio
 * 1/S + K / PageNum has a constant term, so when the sequence is not several
 * times longer than the token budget the scoring costs more than it saves;
 * the first-order rule is PageNum at least a few times the K selected
 * pages).  Host only: returns 1 when a step over sequences of at most
 * max_seq_len tokens should run dense_decode_attention instead, that is
 * when ceil(max_seq_len / S) <= ratio * n_sel; ratio <= 0 takes
 * SPG_DENSE_BYPASS_RATIO, the crossover measured on GB300 for the
 * benchmark's 32-head MHA (128-page budget) and GQA-8 (256-page budget)
 * shapes.  0 otherwise, and 0 when spg_validate rejects p or for SPG_SEL_ALL. */
#define SPG_DENSE_BYPASS_RATIO 2.5f
int32_t spg_prefer_dense(const spg_params* p, int32_t max_seq_len, float ratio);

/* Which kernel(s) sparse_decode_step launches for these parameters (host
 * only; NULL when spg_validate rejects them): "k_fused" (one thread-block
 * cluster per unit), "k_sched" (the persistent scheduled step), or the
 * separate scoring and attention kernels.  A diagnostic for benchmarks and
 * tests; the choice is made by the library (see spg_set_step_kernel). */
const char* spg_step_kernel(const spg_params* p);

/* Kernel launches one sparse_decode_step call makes for these parameters
 * (host only; 0 when spg_validate rejects them). */
int32_t spg_step_launches(const spg_params* p);

/* Process-wide preference between the two single-launch step kernels, for
 * comparing them: 0 = automatic (the cluster kernel where it applies, else
 * the scheduled kernel), 1 = the cluster kernel only, 2 = the scheduled
 * kernel only (shapes it does not take use the separate kernels).  Results
 * are the same up to the order of floating-point sums.  Not thread-safe with respect
 * to launches in flight on other host threads.  SPG_EINVAL for other values. */
spg_status spg_set_step_kernel(int32_t kernel);

/* Waits for `stream`, then copies the workspace error word to *bits. */
spg_status spg_read_device_error(const void* ws, int32_t* bits, spg_stream_t stream);

/* Test hook for the bounded waits.  Arms a one-shot flag in the workspace:
 * the next split-K attention launch on it (sparse_decode_attention,
 * dense_decode_attention, or a step that falls back to them) has its first
 * CTA issue no copy for its first ring stage and never complete it, so the
 * consumer's bounded wait (at most 100 ms) runs out with nothing in flight;
 * the launch then finishes with SPG_DEVERR_TIMEOUT in the error word and
 * its results are not valid (zero the workspace afterwards, as after any
 * timeout).  For testing the error path only.  Asynchronous on `stream`. */
spg_status spg_test_withhold_first_stage(void* ws, spg_stream_t stream);

/* Clears the workspace error word (asynchronous on `stream`). */
spg_status spg_clear_device_error(void* ws, spg_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPG_H_ */
