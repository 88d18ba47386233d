// Page scoring and exact top-k page selection.
//
// Scoring streams one metadata row per candidate page:
//  * Quest (Quest 完全拆解, 核心机制): score = max over the kv-head group's
//    query heads of sum_i max(q_i m_i, q_i M_i) = sum_i q-_i m_i + q+_i M_i
//    (q- = min(q, 0), q+ = max(q, 0)): a [pages x 2d] x [2d x G] product,
//    scored 16 pages at a time on the tensor cores (QuestMma) from rows
//    staged in shared memory by one bulk copy per CTA.
//  * Sketch (SALS长序列推理优化, QSI steps 1-3): the group-mean query is
//    projected through P and quantised to int8 (same fp32 rule as the keys),
//    the int4 key codes are unpacked to int8 lanes and dotted with dp4a
//    (exact int32), dequantised by sq * sk_block / sqrt(d), and reduced to a
//    block log-sum-exp with warp shuffles; one warp per block.
//
// Top-k (SALS QSI Top-k: exact, stable; Day 10·2: lower index wins ties):
// the candidates' scores become order-preserving uint32 keys in shared
// memory.  A radix select finds the k-th largest key: it skips the bits all
// keys share (from the block min and max), then takes 11-bit digits, which
// for spread-out scores settles in one histogram pass.  The keys above the
// threshold plus the lowest-index keys equal to it are compacted in index
// order with two block scans, which yields ascending page ids without a
// sort.  Only int32 page ids reach global memory.  The selection runs in the
// last scoring CTA of each (batch, kv-head) to finish (an arrival counter
// per unit, reset by that CTA), so scoring and selection are one launch;
// very long page tables use a separate selection kernel instead.
#include <float.h>

#include "spg_select_core.cuh"
#include "spg_internal.h"

namespace spg {
namespace {

constexpr int kQuestPagesPerCta = 64;  // 4 warps x one 16-page tile
constexpr int kSketchBlocksPerCta = 8;  // one warp per block
constexpr int kFusedTopkMaxPages = 8192;

struct SelectArgs {
  const void* q;
  const void* k_pool;  // probe selector: the keys it samples
  const int32_t* page_table;
  const int32_t* seq_lens;
  const void* minmax;
  const uint8_t* sketch;
  const float* sketch_scale;
  const float* proj;
  float* scores;      // [B][Hkv][MP]
  int32_t* sel;       // nullptr -> scores only
  int32_t* sel_cnt;
  int32_t* counters;  // [B][Hkv] scoring CTAs done, zero between launches
  int32_t* err;
  int Hkv, G, S, d, MP, n_phys, n_sink, n_recent, n_sel;
  float inv_sqrt_d;
  float top_p, tau;  // adaptive budget (top_p 0: off)
  int min_pages;
  int n_probe;       // probe selector: sampled tokens per page
};

// Selection of one unit from its scores row (global, written by this launch
// or the previous one): forced sinks, the exact top-k candidates (trimmed by
// the adaptive budget when top_p > 0; tps: its shared-memory scratch),
// forced recent pages, then -1 padding; sel_cnt.
template <int MAXN>
__device__ void select_unit(const float* srow, int P, int lo, int hi, int n_sel, int32_t* out,
                            int32_t* cnt_out, uint32_t* s_keys, TopkSmem<MAXN>& t, float top_p,
                            float tau, int min_pages, uint32_t* tps) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int nc = hi - lo, nf = P - nc;
  int k_top = min(max(n_sel - nf, 0), nc);
  for (int i = tid; i < lo; i += nt) out[i] = i;
  if (k_top > 0) {
    if (k_top == nc && top_p <= 0.f) {
      for (int i = tid; i < nc; i += nt) out[lo + i] = lo + i;
    } else {
      for (int i = tid; i < nc; i += nt) s_keys[i] = score_key(__ldcg(srow + lo + i));
      __syncthreads();
      if (k_top == nc)
        for (int i = tid; i < nc; i += nt) out[lo + i] = lo + i;
      else
        block_topk(s_keys, nc, k_top, lo, out + lo, t);
      if (top_p > 0.f) {
        __syncthreads();
        k_top = topp_trim(s_keys, nc, out + lo, k_top, lo, tau, top_p, min_pages, tps,
                          reinterpret_cast<int*>(tps + kTopPScratchWords),
                          reinterpret_cast<float*>(tps + kTopPScratchWords + 40));
      }
    }
  }
  __syncthreads();
  for (int j = tid; j < P - hi; j += nt) out[lo + k_top + j] = hi + j;
  const int count = lo + k_top + (P - hi);
  for (int i = count + tid; i < n_sel; i += nt) out[i] = -1;
  if (tid == 0) *cnt_out = count;
}

// Arrival of a scoring CTA; the last one of its unit selects the unit's pages.
__device__ __forceinline__ void arrive_and_select(const SelectArgs& a, int unit, int P, int lo,
                                                  int hi, uint32_t* s_keys, TopkShared& t,
                                                  int* s_last, uint32_t* tps) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) *s_last = atomicAdd(&a.counters[unit], 1) == static_cast<int>(gridDim.x) - 1;
  __syncthreads();
  if (!*s_last) return;
  __threadfence();
  select_unit(a.scores + static_cast<size_t>(unit) * a.MP, P, lo, hi, a.n_sel,
              a.sel + static_cast<size_t>(unit) * a.n_sel, a.sel_cnt + unit, s_keys, t, a.top_p,
              a.tau, a.min_pages, tps);
  if (threadIdx.x == 0) a.counters[unit] = 0;  // ready for the next call
}

__device__ __forceinline__ int seq_pages(const SelectArgs& a, int b, int* L_out) {
  int L = a.seq_lens[b];
  if (L < 0 || L > a.MP * a.S) {
    if (blockIdx.x == 0 && threadIdx.x == 0) record_error(a.err, SPG_DEVERR_SEQ_LEN);
    L = 0;
  }
  *L_out = L;
  return (L + a.S - 1) / a.S;
}

// Quest scores (+ fused selection): grid (ceil(MP/64), B*Hkv), 128 threads.
// The CTA's 64 metadata rows are one contiguous range (logical page order):
// one bulk copy stages them, then each warp scores one 16-page tile on the
// tensor cores while the next CTAs' copies are in flight.
template <typename T, int D, int G>
__global__ void __launch_bounds__(128) k_quest_select(const SelectArgs a, int fused) {
  constexpr int RB = 2 * D * static_cast<int>(sizeof(T));  // bytes of one metadata row
  extern __shared__ __align__(128) uint8_t smem[];
  T* rows = reinterpret_cast<T*>(smem);                                    // [64][2d]
  uint32_t* s_keys = reinterpret_cast<uint32_t*>(smem + kQuestPagesPerCta * RB);  // fused top-k
  __shared__ __align__(8) uint64_t bar;
  __shared__ TopkShared s_t;
  __shared__ int s_last;

  pdl_wait();
  const int unit = blockIdx.y, Hkv = a.Hkv;
  const int b = unit / Hkv, h = unit % Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int p0 = blockIdx.x * kQuestPagesPerCta;
  int L;
  const int P = seq_pages(a, b, &L);
  const int lo = min(a.n_sink, P), hi = max(P - a.n_recent, lo);
  const int n_rows = max(0, min(kQuestPagesPerCta, P - p0));
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bar, static_cast<uint32_t>(n_rows) * RB);
    if (n_rows > 0)
      bulk_g2s(rows,
               static_cast<const T*>(a.minmax) + (static_cast<size_t>(unit) * a.MP + p0) * 2 * D,
               static_cast<uint32_t>(n_rows) * RB, &bar);
  }
  QuestMma<T, D, G> qm;
  qm.init(static_cast<const T*>(a.q) + (static_cast<size_t>(b) * Hkv * G + h * G) * D, lane);
  if (!mbar_wait_bounded(&bar, 0)) {
    if (lane == 0) record_error(a.err, SPG_DEVERR_TIMEOUT);
    mbar_wait_bounded(&bar, 0);  // drain before the CTA may leave
  }
  float s0, s1;
  qm.tile(rows + warp * 16 * 2 * D, p0 + warp * 16, lane, s0, s1);
  if ((lane & 3) == 0) {
    const int g = lane >> 2;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int p = p0 + warp * 16 + g + 8 * half;
      if (p < a.MP)
        a.scores[static_cast<size_t>(unit) * a.MP + p] =
            (p >= lo && p < hi) ? (half ? s1 : s0) : -INFINITY;
    }
  }
  pdl_trigger();
  if (fused) arrive_and_select(a, unit, P, lo, hi, s_keys, s_t, &s_last, reinterpret_cast<uint32_t*>(rows));
}

// Sketch scores (+ fused selection): grid (ceil(MP/8), B*Hkv), 256 threads,
// one warp per block; ds = 16 (8 bytes of codes per token).
template <typename TQ>
__global__ void __launch_bounds__(256) k_sketch_select(const SelectArgs a, int fused) {
  constexpr int DS = 16;
  extern __shared__ __align__(128) uint32_t s_keys[];  // 16-byte key loads
  __shared__ float s_qbar[256];
  __shared__ float s_P[256 * DS];
  __shared__ int s_qc[4];  // packed int8 codes: even 0-6, odd 1-7, even 8-14, odd 9-15
  __shared__ float s_sq;
  __shared__ TopkShared s_t;
  __shared__ int s_last;

  pdl_wait();
  const int unit = blockIdx.y, Hkv = a.Hkv, G = a.G, d = a.d, S = a.S;
  const int b = unit / Hkv, h = unit % Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int blk = blockIdx.x * kSketchBlocksPerCta + warp;
  int L;
  const int P = seq_pages(a, b, &L);
  const int lo = min(a.n_sink, P), hi = max(P - a.n_recent, lo);
  const int ph = (blk >= lo && blk < hi) ? blk : -1;  // candidate (logical block)
  // this warp's block codes and scale, in flight while the index query is built
  const size_t lrow = static_cast<size_t>(unit) * a.MP + (ph < 0 ? 0 : ph);
  const size_t row0 = lrow * S;
  uint2 wk[4];
  float sk = 1.f;
  if (ph >= 0) {
    sk = __ldg(a.sketch_scale + lrow);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int t = lane + 32 * k;
      if (t < S) wk[k] = __ldg(reinterpret_cast<const uint2*>(a.sketch + (row0 + t) * (DS / 2)));
    }
  }

  sketch_index_query<TQ>(static_cast<const TQ*>(a.q) + (static_cast<size_t>(b) * Hkv * G + h * G) * d,
                         G, d, a.proj, s_qbar, s_P, s_qc, &s_sq);
  if (blk < a.MP) {
    float score = -INFINITY;
    if (ph >= 0)
      score = sketch_block_score(wk, S, s_qc, __fmul_rn(__fmul_rn(s_sq, sk), a.inv_sqrt_d));
    if (lane == 0) a.scores[static_cast<size_t>(unit) * a.MP + blk] = score;
  }
  pdl_trigger();
  if (fused) arrive_and_select(a, unit, P, lo, hi, s_keys, s_t, &s_last, reinterpret_cast<uint32_t*>(s_P));
}

// Probe scores (+ fused selection; Day 10·2 sparse top-k, §1-§2): grid
// (ceil(MP / 32), B*Hkv), 128 threads, one warp per page at a time (8 pages
// per warp).  A page's score is the largest q . k over its sampled tokens:
// from the page's first token in steps of max(valid / n_probe, 1), the max
// also over the group's G query rows.  Each sampled key row (d elements,
// contiguous) is one coalesced warp load; a warp keeps up to 8 rows in
// flight; q in registers (d / 32 channels per lane, fp32); dot products
// summed over the warp by shuffles.
constexpr int kProbePagesPerCta = 32;
constexpr int kProbeMaxInFlight = 8;

template <typename T, int D, int G>
__global__ void __launch_bounds__(128) k_probe_select(const SelectArgs a, int fused) {
  constexpr int CPL = D / 32;  // channels per lane
  extern __shared__ __align__(128) uint32_t s_keys[];
  __shared__ TopkShared s_t;
  __shared__ int s_last;
  __shared__ __align__(16) uint32_t s_scratch[kTopPScratchWords + 80];
  pdl_wait();
  const int unit = blockIdx.y, Hkv = a.Hkv, S = a.S;
  const int b = unit / Hkv, h = unit % Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int L;
  const int P = seq_pages(a, b, &L);
  const int lo = min(a.n_sink, P), hi = max(P - a.n_recent, lo);
  float qf[G][CPL];
  const T* qb = static_cast<const T*>(a.q) + (static_cast<size_t>(b) * Hkv * G + h * G) * D;
#pragma unroll
  for (int g = 0; g < G; ++g) load_cvt<T, CPL>(qb + g * D + lane * CPL, qf[g]);
  const int n_probe = max(a.n_probe, 1);
  for (int j = warp; j < kProbePagesPerCta; j += 4) {
    const int p = blockIdx.x * kProbePagesPerCta + j;
    if (p >= a.MP) break;
    float score = -INFINITY;
    if (p >= lo && p < hi) {  // a candidate page
      const int phys = a.page_table[static_cast<size_t>(b) * a.MP + p];
      if (phys < 0 || phys >= a.n_phys) {
        if (lane == 0) record_error(a.err, SPG_DEVERR_PAGE_ID);
      } else {
        const int valid = min(S, L - p * S);
        const int step = max(valid / n_probe, 1);
        const T* page = static_cast<const T*>(a.k_pool) + (static_cast<size_t>(phys) * Hkv + h) * S * D;
        for (int t0 = 0; t0 < valid; t0 += step * kProbeMaxInFlight) {
          float kf[kProbeMaxInFlight][CPL];
#pragma unroll
          for (int r = 0; r < kProbeMaxInFlight; ++r) {
            const int t = t0 + r * step;
            if (t < valid) load_cvt<T, CPL>(page + static_cast<size_t>(t) * D + lane * CPL, kf[r]);
          }
#pragma unroll
          for (int r = 0; r < kProbeMaxInFlight; ++r) {
            const int t = t0 + r * step;
            if (t < valid) {  // warp-uniform
#pragma unroll
              for (int g = 0; g < G; ++g) {
                float acc = 0.f;
#pragma unroll
                for (int c = 0; c < CPL; ++c) acc = fmaf(qf[g][c], kf[r][c], acc);
                acc = warp_sum(acc);
                score = fmaxf(score, acc);
              }
            }
          }
        }
      }
    }
    if (lane == 0) a.scores[static_cast<size_t>(unit) * a.MP + p] = score;
  }
  pdl_trigger();
  if (fused) arrive_and_select(a, unit, P, lo, hi, s_keys, s_t, &s_last, s_scratch);
}

// Selection alone, for page tables too long to select inside the scoring
// launch: one CTA (1024 threads) per (batch, kv-head).
__global__ void __launch_bounds__(1024) k_topk(const SelectArgs a) {
  extern __shared__ __align__(128) uint32_t s_keys[];  // 16-byte key loads
  __shared__ TopkSmem<kMaxTopkPages> s_t;
  pdl_wait();
  const int unit = blockIdx.x;
  const int b = unit / a.Hkv;
  int L = a.seq_lens[b];
  if (L < 0 || L > a.MP * a.S) L = 0;  // recorded by the scoring kernel
  const int P = (L + a.S - 1) / a.S;
  const int lo = min(a.n_sink, P), hi = max(P - a.n_recent, lo);
  pdl_trigger();
  select_unit(a.scores + static_cast<size_t>(unit) * a.MP, P, lo, hi, a.n_sel,
              a.sel + static_cast<size_t>(unit) * a.n_sel, a.sel_cnt + unit, s_keys, s_t, 0.f, 1.f,
              0, nullptr);  // the adaptive budget is limited to tables of <= 8192 pages
}

// The sketch selector's integer arithmetic laid bare (QSI steps 1-2): per
// unit, the int8 index query (the same warp routine every scan uses) and the
// exact int32 dot of the query codes with every token of every candidate
// block (the same token routine as the block scores).  Grid: one CTA of 256
// threads per (batch, kv-head).
template <typename TQ>
__global__ void __launch_bounds__(256) k_sketch_dots(const SelectArgs a, int32_t* qc_out,
                                                      float* sq_out, int32_t* dots) {
  constexpr int DS = 16;
  __shared__ float s_qbar[256];
  __shared__ float s_P[256 * DS];
  __shared__ int s_qc[4];
  __shared__ int s_bias;
  pdl_wait();
  const int unit = blockIdx.x, Hkv = a.Hkv, G = a.G, d = a.d, S = a.S;
  const int b = unit / Hkv, h = unit % Hkv;
  int L;
  const int P = seq_pages(a, b, &L);
  const int lo = min(a.n_sink, P), hi = max(P - a.n_recent, lo);
  for (int i = threadIdx.x; i < d * DS; i += blockDim.x) s_P[i] = a.proj[i];
  __syncthreads();
  if (threadIdx.x < 32) {
    int qc4[4], code;
    float sq;
    sketch_index_query_warp<TQ>(static_cast<const TQ*>(a.q) + (static_cast<size_t>(b) * Hkv * G + h * G) * d,
                                G, d, s_P, s_qbar, threadIdx.x, qc4, sq, &code);
    if (threadIdx.x < DS) qc_out[static_cast<size_t>(unit) * DS + threadIdx.x] = code;
    if (threadIdx.x == 0) {
      sq_out[unit] = sq;
#pragma unroll
      for (int k = 0; k < 4; ++k) s_qc[k] = qc4[k];
      s_bias = sketch_query_bias(qc4);
    }
  }
  __syncthreads();
  const int qc[4] = {s_qc[0], s_qc[1], s_qc[2], s_qc[3]};
  const int bias = s_bias;
  const size_t base = static_cast<size_t>(unit) * a.MP * S;
  for (size_t i = threadIdx.x; i < static_cast<size_t>(a.MP) * S; i += blockDim.x) {
    const int blk = static_cast<int>(i / S);
    int v = 0;
    if (blk >= lo && blk < hi)
      v = sketch_token_dot(__ldg(reinterpret_cast<const uint2*>(a.sketch + (base + i) * (DS / 2))), qc, bias);
    dots[base + i] = v;
  }
}

template <typename T>
cudaError_t probe_typed(const spg_params& p, const SelectArgs& a, int fused, size_t smem_keys,
                        cudaStream_t st) {
  dim3 grid((p.max_pages_per_seq + kProbePagesPerCta - 1) / kProbePagesPerCta,
            p.batch * p.num_kv_heads);
  const int G = a.G;
#define SPG_PS(D_, G_)                                          \
  if (p.head_dim == D_ && G == G_) {                             \
    auto kern = k_probe_select<T, D_, G_>;                       \
    cudaError_t e = ensure_smem(kern, smem_keys);                \
    if (e != cudaSuccess) return e;                              \
    return launch_pdl(kern, grid, dim3(128), smem_keys, st, a, fused); \
  }
  SPG_PS(128, 1) SPG_PS(128, 2) SPG_PS(128, 4) SPG_PS(128, 8)
  SPG_PS(64, 1) SPG_PS(64, 2) SPG_PS(64, 4) SPG_PS(64, 8)
#undef SPG_PS
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t quest_typed(const spg_params& p, const SelectArgs& a, int fused, size_t smem_keys,
                        cudaStream_t st) {
  dim3 grid((p.max_pages_per_seq + kQuestPagesPerCta - 1) / kQuestPagesPerCta,
            p.batch * p.num_kv_heads);
  const int G = a.G;
  const size_t smem = static_cast<size_t>(kQuestPagesPerCta) * 2 * p.head_dim * sizeof(T) + smem_keys;
#define SPG_QS(D_, G_)                                                                     \
  if (p.head_dim == D_ && G == G_) {                                                        \
    auto kern = k_quest_select<T, D_, G_>;                                                  \
    cudaError_t e = ensure_smem(kern, smem);                                                \
    if (e != cudaSuccess) return e;                                                         \
    return launch_pdl(kern, grid, dim3(128), smem, st, a, fused);                           \
  }
  SPG_QS(128, 1) SPG_QS(128, 2) SPG_QS(128, 4) SPG_QS(128, 8)
  SPG_QS(64, 1) SPG_QS(64, 2) SPG_QS(64, 4) SPG_QS(64, 8)
#undef SPG_QS
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_select(const spg_params& p, const void* q, const int32_t* page_table,
                          const int32_t* seq_lens, const void* minmax, const uint8_t* sketch,
                          const float* sketch_scale, const float* proj, float* scores,
                          int32_t* sel, int32_t* sel_cnt, const Workspace& ws,
                          cudaStream_t stream) {
  SelectArgs a{};
  a.q = q;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.minmax = minmax;
  a.sketch = sketch;
  a.sketch_scale = sketch_scale;
  a.proj = proj;
  a.scores = scores;
  a.sel = sel;
  a.sel_cnt = sel_cnt;
  a.counters = ws.sel_counters;
  a.err = ws.err;
  a.Hkv = p.num_kv_heads;
  a.G = p.num_q_heads / p.num_kv_heads;
  a.S = p.page_size;
  a.d = p.head_dim;
  a.MP = p.max_pages_per_seq;
  a.n_phys = p.num_phys_pages;
  a.n_sink = p.n_sink_pages;
  a.n_recent = p.n_recent_pages;
  a.n_sel = n_sel_pages(p);
  a.inv_sqrt_d = 1.0f / sqrtf(static_cast<float>(p.head_dim));
  a.top_p = p.top_p;
  a.min_pages = p.min_pages;
  a.tau = p.selector == SPG_SEL_SKETCH_INT4
              ? 1.0f  // a log block mass; Quest and probe scores are dot products
              : (p.softmax_scale > 0.f ? p.softmax_scale : 1.0f / sqrtf(static_cast<float>(p.head_dim)));
  a.n_probe = p.n_probe > 0 ? p.n_probe : kDefaultProbes;
  a.k_pool = minmax;  // the probe selector samples the keys themselves
  const int fused = (sel != nullptr && p.max_pages_per_seq <= kFusedTopkMaxPages) ? 1 : 0;
  const size_t smem = fused ? sizeof(uint32_t) * p.max_pages_per_seq : 0;
  cudaError_t e;
  if (p.selector == SPG_SEL_PROBE) {
    e = p.kv_dtype == SPG_F16 ? probe_typed<__half>(p, a, fused, smem, stream)
                              : probe_typed<__nv_bfloat16>(p, a, fused, smem, stream);
  } else if (p.selector == SPG_SEL_QUEST) {
    // the metadata's type: the pool's, or the query's for int8 pools
    const int meta = p.kv_dtype == SPG_I8 ? p.q_dtype : p.kv_dtype;
    e = meta == SPG_F16 ? quest_typed<__half>(p, a, fused, smem, stream)
                        : quest_typed<__nv_bfloat16>(p, a, fused, smem, stream);
  } else {
    dim3 grid((p.max_pages_per_seq + kSketchBlocksPerCta - 1) / kSketchBlocksPerCta,
              p.batch * p.num_kv_heads);
    if (p.q_dtype == SPG_F16) {
      auto kern = k_sketch_select<__half>;
      e = ensure_smem(kern, smem);
      if (e == cudaSuccess)
        e = launch_pdl(kern, grid, dim3(kSketchBlocksPerCta * 32), smem, stream, a, fused);
    } else {
      auto kern = k_sketch_select<__nv_bfloat16>;
      e = ensure_smem(kern, smem);
      if (e == cudaSuccess)
        e = launch_pdl(kern, grid, dim3(kSketchBlocksPerCta * 32), smem, stream, a, fused);
    }
  }
  if (e != cudaSuccess || sel == nullptr || fused) return e;
  const size_t tsmem = sizeof(uint32_t) * p.max_pages_per_seq;
  e = ensure_smem(k_topk, tsmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_topk, dim3(p.batch * p.num_kv_heads), dim3(1024), tsmem, stream, a);
}

}  // namespace spg

namespace spg {

cudaError_t launch_sketch_dots(const spg_params& p, const void* q, const int32_t* seq_lens,
                               const uint8_t* sketch, const float* proj, int32_t* qc, float* sq,
                               int32_t* dots, int32_t* err, cudaStream_t stream) {
  SelectArgs a{};
  a.q = q;
  a.seq_lens = seq_lens;
  a.sketch = sketch;
  a.proj = proj;
  a.err = err;
  a.Hkv = p.num_kv_heads;
  a.G = p.num_q_heads / p.num_kv_heads;
  a.S = p.page_size;
  a.d = p.head_dim;
  a.MP = p.max_pages_per_seq;
  a.n_sink = p.n_sink_pages;
  a.n_recent = p.n_recent_pages;
  const dim3 grid(p.batch * p.num_kv_heads);
  if (p.q_dtype == SPG_F16)
    return launch_pdl(k_sketch_dots<__half>, grid, dim3(256), 0, stream, a, qc, sq, dots);
  return launch_pdl(k_sketch_dots<__nv_bfloat16>, grid, dim3(256), 0, stream, a, qc, sq, dots);
}

}  // namespace spg
